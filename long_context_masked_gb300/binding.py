"""ctypes binding of the C ABI in ``include/lca.h`` (argument marshalling only).

Torch tensors provide device memory and the current CUDA stream; every step of the
computation runs in the library's kernels.  Nothing here falls back to another
implementation: if the library is missing or a call fails, an ``LcaError`` is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import inputs as I

_PKG = os.path.dirname(os.path.abspath(__file__))

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "cuda error", 4: "out of memory",
          5: "timeout", 6: "plan mismatch"}


class LcaError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status})")
        self.status = status


class MaskDescC(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int32), ("seqlen", ctypes.c_int32),
                ("window", ctypes.c_int32), ("num_global", ctypes.c_int32),
                ("prefix_len", ctypes.c_int32), ("block", ctypes.c_int32),
                ("base_causal", ctypes.c_int32), ("num_segments", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p), ("map_heads", ctypes.c_int32),
                ("n_row_blocks", ctypes.c_int32), ("n_col_blocks", ctypes.c_int32),
                ("row_block_offsets", ctypes.c_void_p), ("col_block_offsets", ctypes.c_void_p),
                ("block_map", ctypes.c_void_p)]


class ShapeC(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seqlen", ctypes.c_int32), ("h_q", ctypes.c_int32),
                ("h_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("q_row_stride", ctypes.c_int64), ("k_row_stride", ctypes.c_int64),
                ("v_row_stride", ctypes.c_int64), ("o_row_stride", ctypes.c_int64),
                ("do_row_stride", ctypes.c_int64), ("dq_row_stride", ctypes.c_int64),
                ("dk_row_stride", ctypes.c_int64), ("dv_row_stride", ctypes.c_int64)]


class PlanInfoC(ctypes.Structure):
    _fields_ = [("seqlen", ctypes.c_int32), ("tile_q", ctypes.c_int32), ("tile_k", ctypes.c_int32),
                ("n_qt", ctypes.c_int32), ("n_kt", ctypes.c_int32), ("map_heads", ctypes.c_int32),
                ("mask_type", ctypes.c_int32), ("nnz", ctypes.c_int64),
                ("n_partial", ctypes.c_int64), ("device_bytes", ctypes.c_int64)]


class KernelTimeC(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


_lib = None


def library_path() -> str:
    return os.path.join(_PKG, "_lib", "liblca.so")


def load_library():
    """Load liblca.so (built by ``long_context_masked_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise LcaError(f"CUDA library not built ({path}); run long_context_masked_gb300.build", 3)
    lib = ctypes.CDLL(path)
    vp, i32, u64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_float
    sig = {
        "lca_mask_build": ([ctypes.POINTER(MaskDescC), ctypes.c_int, ctypes.c_int, vp,
                            ctypes.POINTER(vp)], i32),
        "lca_plan_get_info": ([vp, ctypes.POINTER(PlanInfoC)], i32),
        "lca_plan_export": ([vp] + [vp] * 10, i32),
        "lca_plan_destroy": ([vp], None),
        "lca_attn_fwd": ([vp, ctypes.POINTER(ShapeC), vp, vp, vp, vp, vp, f32, vp], i32),
        "lca_attn_bwd_workspace": ([vp, ctypes.POINTER(ShapeC), ctypes.c_int], ctypes.c_size_t),
        "lca_attn_bwd": ([vp, ctypes.POINTER(ShapeC)] + [vp] * 10 +
                         [ctypes.c_size_t, f32, ctypes.c_int, vp], i32),
        "lca_get_last_device_error": ([vp], i32),
        "lca_set_wait_timeout_ns": ([u64], None),
        "lca_selftest_wait_timeout": ([u64, vp], i32),
        "lca_selftest_umma": ([ctypes.c_int, vp, vp, vp, vp], i32),
        "lca_status_string": ([i32], ctypes.c_char_p),
        "lca_attn_bwd_noalloc": ([vp, ctypes.POINTER(ShapeC)] + [vp] * 9 + [f32, vp], i32),
        "lca_profile_enable": ([ctypes.c_int], None),
        "lca_block_scores_workspace": ([ctypes.POINTER(ShapeC), ctypes.c_int, ctypes.c_int],
                                       ctypes.c_size_t),
        "lca_block_scores": ([ctypes.POINTER(ShapeC), vp, vp, ctypes.c_int, ctypes.c_int, f32, vp,
                              vp, ctypes.c_size_t, vp], i32),
        "lca_block_topk": ([vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp],
                           i32),
        "lca_profile_read": ([ctypes.POINTER(KernelTimeC), ctypes.c_int], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(what: str, status: int):
    if status != 0:
        raise LcaError(what, status)


def _stream(stream) -> Optional[int]:
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _dev_array(arr, dtype, device):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(np.asarray(arr, dtype=dtype)))
    return t.to(device)


class Plan:
    """A tile plan (owns its device buffers; freed when garbage collected)."""

    def __init__(self, handle: int, desc: I.MaskDesc):
        self._h = ctypes.c_void_p(handle)
        self.desc = desc
        info = PlanInfoC()
        _check("lca_plan_get_info", load_library().lca_plan_get_info(self._h, ctypes.byref(info)))
        self.info = {k: getattr(info, k) for k, _ in PlanInfoC._fields_}

    @property
    def handle(self):
        return self._h

    def export(self) -> dict:
        """Host copies of every plan array.  ``cls`` holds the tile bytes (class in bits 0-1,
        empty-half flags above: inputs.TILE_*), ``kt_cls`` / ``qt_cls`` the list entries."""
        inf = self.info
        hm, nq, nk, nnz = inf["map_heads"], inf["n_qt"], inf["n_kt"], inf["nnz"]
        out = {"cls": np.zeros(hm * nq * nk, np.uint8), "rowptr": np.zeros(hm * nq + 1, np.int32),
               "kt_idx": np.zeros(nnz, np.int32), "kt_cls": np.zeros(nnz, np.uint8),
               "colptr": np.zeros(hm * nk + 1, np.int32), "qt_idx": np.zeros(nnz, np.int32),
               "qt_cls": np.zeros(nnz, np.uint8), "work_q": np.zeros(hm * nq, np.int32),
               "work_k": np.zeros(hm * nk, np.int32), "n_valid": np.zeros(hm, np.int64)}
        order = ["cls", "rowptr", "kt_idx", "kt_cls", "colptr", "qt_idx", "qt_cls", "work_q",
                 "work_k", "n_valid"]
        ptrs = [out[k].ctypes.data_as(ctypes.c_void_p) if out[k].size else None for k in order]
        _check("lca_plan_export", load_library().lca_plan_export(self._h, *ptrs))
        out["cls"] = out["cls"].reshape(hm, nq, nk)
        return out

    def n_valid(self) -> np.ndarray:
        """Allowed (i, j) pairs per map head (int64 [map_heads]); copies nothing else."""
        nv = np.zeros(self.info["map_heads"], np.int64)
        _check("lca_plan_export", load_library().lca_plan_export(
            self._h, *([None] * 9), nv.ctypes.data_as(ctypes.c_void_p)))
        return nv

    def __del__(self):
        if getattr(self, "_h", None) is not None and self._h.value and _lib is not None:
            _lib.lca_plan_destroy(self._h)
            self._h = None


def mask_build(desc: I.MaskDesc, tile_q: int = 128, tile_k: int = 128, stream=None,
               device: str = "cuda") -> Plan:
    """Build the tile plan of ``desc`` on the GPU (lca_mask_build)."""
    lib = load_library()
    keep = []
    c = MaskDescC()
    c.type, c.seqlen = desc.type, desc.seqlen
    c.window, c.num_global, c.prefix_len = desc.window, desc.num_global, desc.prefix_len
    c.block, c.base_causal = desc.block, desc.base_causal
    if desc.cu_seqlens is not None:
        t = _dev_array(desc.cu_seqlens, np.int32, device)
        keep.append(t)
        c.num_segments = len(desc.cu_seqlens) - 1
        c.cu_seqlens = t.data_ptr()
    c.map_heads = desc.map_heads
    if desc.block_map is not None:
        bm = desc.block_map
        if hasattr(bm, "data_ptr") and getattr(bm, "is_cuda", False):
            # a device map (e.g. from block_topk) is passed as is
            import torch

            if bm.dtype != torch.uint8 or not bm.is_contiguous() or bm.dim() != 3:
                raise LcaError("block_map: contiguous uint8 [map_heads, n_rb, n_cb] expected", 1)
            t = bm
        else:
            bm = np.asarray(bm, np.uint8)
            t = _dev_array(bm, np.uint8, device)
        keep.append(t)
        c.block_map = t.data_ptr()
        c.n_row_blocks, c.n_col_blocks = int(bm.shape[1]), int(bm.shape[2])
    for name in ("row_offsets", "col_offsets"):
        arr = getattr(desc, name)
        if arr is not None:
            t = _dev_array(arr, np.int32, device)
            keep.append(t)
            setattr(c, "row_block_offsets" if name == "row_offsets" else "col_block_offsets",
                    t.data_ptr())
    out = ctypes.c_void_p()
    st = lib.lca_mask_build(ctypes.byref(c), tile_q, tile_k, _stream(stream), ctypes.byref(out))
    _check("lca_mask_build", st)
    return Plan(out.value, desc)


def _shape(q, k, v, o, do=None, dq=None, dk=None, dv=None):
    """lca_shape of the given tensors.  Each tensor is [B, S, heads, d] with packed heads
    and its own row stride (slices of a packed QKV tensor are fine); the gradient-side
    strides are filled from dO/dQ/dK/dV when they are given."""
    b, s, hq, d = q.shape
    hkv = k.shape[2]
    named = (("q", q, hq), ("k", k, hkv), ("v", v, hkv), ("o", o, hq), ("do", do, hq),
             ("dq", dq, hq), ("dk", dk, hkv), ("dv", dv, hkv))
    for name, t, h in named:
        if t is None:
            continue
        if t.stride(3) != 1 or t.stride(2) != d or t.stride(0) != s * t.stride(1):
            raise LcaError(f"{name}: unsupported layout {tuple(t.stride())}", 1)
        if tuple(t.shape[:2]) != (b, s) or t.shape[2] != h or t.shape[3] != d:
            raise LcaError(f"{name}: shape {tuple(t.shape)}", 1)
        if t.device != q.device:
            raise LcaError(f"{name}: on {t.device}, q on {q.device}", 1)
    sh = ShapeC(b, s, hq, hkv, d, q.stride(1), k.stride(1), v.stride(1), o.stride(1))
    for name, t, _ in named[4:]:
        if t is not None:
            setattr(sh, f"{name}_row_stride", t.stride(1))
    return sh


def attn_fwd(plan: Plan, q, k, v, scale: Optional[float] = None, out=None, lse=None,
             stream=None):
    """O and LSE (lca_attn_fwd).  q [B,S,Hq,128], k/v [B,S,Hkv,128] bf16 on the GPU."""
    import torch

    lib = load_library()
    b, s, hq, d = q.shape
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((b, hq, s), dtype=torch.float32, device=q.device) if lse is None else lse
    sh = _shape(q, k, v, o)
    st = lib.lca_attn_fwd(plan.handle, ctypes.byref(sh), q.data_ptr(), k.data_ptr(),
                          v.data_ptr(), o.data_ptr(), l.data_ptr(),
                          float(scale) if scale else 0.0, _stream(stream))
    _check("lca_attn_fwd", st)
    return o, l


def attn_bwd(plan: Plan, q, k, v, o, do, lse, scale: Optional[float] = None, dq=None, dk=None,
             dv=None, workspace=None, stream=None):
    """dQ, dK, dV (lca_attn_bwd)."""
    import torch

    lib = load_library()
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    sh = _shape(q, k, v, o, do, dq, dk, dv)
    ws_bytes = lib.lca_attn_bwd_workspace(plan.handle, ctypes.byref(sh), 0)
    if workspace is None:
        workspace = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=q.device)
    st = lib.lca_attn_bwd(plan.handle, ctypes.byref(sh), q.data_ptr(), k.data_ptr(),
                          v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                          workspace.numel() * workspace.element_size(),
                          float(scale) if scale else 0.0, 0, _stream(stream))
    _check("lca_attn_bwd", st)
    return dq, dk, dv


def attn_bwd_noalloc(plan: Plan, q, k, v, o, do, lse, scale: Optional[float] = None, dq=None,
                     dk=None, dv=None, stream=None):
    """dQ, dK, dV through lca_attn_bwd_noalloc: the backward for callers that cannot
    allocate device memory at that point; its workspace is the library's fixed
    built-in buffer (batch * h_q * round_up(seqlen, 128) <= 2^23).  Pass preallocated dq/dk/dv to
    keep the call free of allocations on the Python side too."""
    import torch

    lib = load_library()
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    sh = _shape(q, k, v, o, do, dq, dk, dv)
    st = lib.lca_attn_bwd_noalloc(plan.handle, ctypes.byref(sh), q.data_ptr(), k.data_ptr(),
                                  v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                                  dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                  float(scale) if scale else 0.0, _stream(stream))
    _check("lca_attn_bwd_noalloc", st)
    return dq, dk, dv


def last_device_error(stream=None) -> int:
    """Status of the bounded device waits since the previous call (0 = ok, 5 = timeout)."""
    return load_library().lca_get_last_device_error(_stream(stream))


def selftest_umma(variant: int, a, b, stream=None):
    import torch

    c = torch.empty((128, 128), dtype=torch.float32, device=a.device)
    _check("lca_selftest_umma", load_library().lca_selftest_umma(
        variant, a.data_ptr(), b.data_ptr(), c.data_ptr(), _stream(stream)))
    return c


def selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    return load_library().lca_selftest_wait_timeout(timeout_ns, _stream(stream))


def profile_enable(on: bool = True):
    """Record CUDA events around every kernel launch of the library."""
    load_library().lca_profile_enable(1 if on else 0)


def profile_read() -> dict:
    """{kernel name: (launches, total ms)} since the last read (synchronises)."""
    buf = (KernelTimeC * 16)()
    n = load_library().lca_profile_read(buf, 16)
    if n < 0:
        raise LcaError("lca_profile_read", 3)
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n)}


def block_scores(q, k, block: int, map_heads: int, scale: Optional[float] = None, out=None,
                 workspace=None, stream=None):
    """fp32 [map_heads, n_b, n_b] block scores from mean-pooled Q and K (lca_block_scores).
    q [1, S, Hq, 128], k [1, S, Hkv, 128] bf16 on the GPU; n_b = ceil(S / block)."""
    import torch

    lib = load_library()
    b, s, hq, d = q.shape
    hkv = k.shape[2]
    sh = ShapeC(b, s, hq, hkv, d, q.stride(1), k.stride(1), k.stride(1), q.stride(1))
    nb = (s + block - 1) // block
    scores = torch.empty((map_heads, nb, nb), dtype=torch.float32, device=q.device) \
        if out is None else out
    ws_bytes = lib.lca_block_scores_workspace(ctypes.byref(sh), block, map_heads)
    if workspace is None:
        workspace = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=q.device)
    st = lib.lca_block_scores(ctypes.byref(sh), q.data_ptr(), k.data_ptr(), block, map_heads,
                              float(scale) if scale else 0.0, scores.data_ptr(),
                              workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                              _stream(stream))
    _check("lca_block_scores", st)
    return scores


def block_topk(scores, k: int, out=None, stream=None):
    """uint8 block map of the k best key blocks of every row of ``scores`` (lca_block_topk):
    descending score, ties by ascending key block.  scores fp32 [H_m, n_rb, n_cb] on the GPU."""
    import torch

    lib = load_library()
    if scores.dtype != torch.float32 or not scores.is_contiguous() or scores.dim() != 3:
        raise LcaError("scores: contiguous fp32 [map_heads, n_rb, n_cb] expected", 1)
    hm, nr, nc = scores.shape
    m = torch.empty((hm, nr, nc), dtype=torch.uint8, device=scores.device) if out is None else out
    st = lib.lca_block_topk(scores.data_ptr(), hm, nr, nc, int(k), m.data_ptr(), _stream(stream))
    _check("lca_block_topk", st)
    return m
