"""ctypes binding of libqnre (include/qnre.h).  Argument marshalling only.

The names follow the C ABI: `qnre_forward`, `qnre_forward_noalloc`,
`ulysses_pack_head_chunk`, `ulysses_merge_output_head_chunk`,
`ulysses_scatter_heads`, `ulysses_gather_heads`,
`ulysses_pack_output_sequence_chunk`, `ulysses_gather_output_head_chunk`,
`ulysses_scatter_qkv_head_chunk`, plus the `Plan` wrapper around
`qnre_plan_create` / `qnre_plan_destroy`.  Tensors are torch CUDA tensors;
torch supplies device memory and the current stream, nothing else.  Every
failure status raises `QnreError`; a missing library raises at first use.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Dict, List, Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqnre.so")
DEBUG_LIB_PATH = os.path.join(HERE, "libqnre_debug.so")  # QNRE_LIB=<this path> selects it
HEADER = os.path.join(os.path.dirname(HERE), "include", "qnre.h")

QNRE_OK = 0
STATUS_NAMES = {
    0: "QNRE_OK", 1: "QNRE_ERR_INVALID_ARG", 2: "QNRE_ERR_UNSUPPORTED", 3: "QNRE_ERR_ALIGNMENT",
    4: "QNRE_ERR_ALIAS", 5: "QNRE_ERR_CAPACITY", 6: "QNRE_ERR_CUDA", 7: "QNRE_ERR_DEVICE",
}
LAYOUTS = {"bshd": 0, "fused": 1}
ROPE_STYLES = {"rotate_half": 0, "interleaved": 1}
FLAG_EPILOGUE_OFF = 0x1
FLAG_W_MULTICAST = 0x2
FLAG_ONE_PAIR = 0x4
DEVICE_BAD_POSITION = 0x1
DEVICE_WAIT_TIMEOUT = 0x2
DEVICE_READY_TIMEOUT = 0x4
DEVICE_BOUNDS = 0x8
HEAD_DIM = 128


class QnreError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class _Out(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("fused", ctypes.c_void_p)]


class _PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("device", "pairs_per_cluster", "clusters", "sms", "row_tiles",
                                            "col_tiles", "work_items", "half_items", "launches")]


class _Tensor4(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("shape", ctypes.c_int64 * 4),
                ("stride", ctypes.c_int64 * 4), ("dtype", ctypes.c_int32)]


_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libqnre.so (built by ulysses_qkv_proj_gb300.build), or the library the
    QNRE_LIB environment variable names (the debug build); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("QNRE_LIB") or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libqnre.so not built ({path}); run `python -m ulysses_qkv_proj_gb300.build`")
    lib = ctypes.CDLL(path)
    c_int, c_i64, c_vp, c_uint = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint
    lib.qnre_status_string.restype = ctypes.c_char_p
    lib.qnre_status_string.argtypes = [c_int]
    lib.qnre_plan_create.restype = c_int
    lib.qnre_plan_create.argtypes = [ctypes.POINTER(c_vp), c_int, c_int, c_int, c_int, c_int, c_i64, c_int, c_uint]
    lib.qnre_plan_destroy.restype = c_int
    lib.qnre_plan_destroy.argtypes = [c_vp]
    lib.qnre_plan_reserve_sms.restype = c_int
    lib.qnre_plan_reserve_sms.argtypes = [c_vp, c_int]
    lib.qnre_plan_describe.restype = c_int
    lib.qnre_plan_describe.argtypes = [c_vp, c_int, c_int, ctypes.POINTER(_PlanInfo)]
    lib.qnre_forward.restype = c_int
    lib.qnre_forward.argtypes = [c_vp, c_int, c_int, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp,
                                 ctypes.POINTER(_Out), c_vp]
    lib.qnre_plan_device_status.restype = c_int
    lib.qnre_plan_device_status.argtypes = [c_vp, c_vp, ctypes.POINTER(c_uint), c_int]
    lib.qnre_debug_bounds.restype = c_int
    lib.qnre_debug_bounds.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), c_int]
    lib.ulysses_pack_head_chunk.restype = c_int
    lib.ulysses_pack_head_chunk.argtypes = [ctypes.POINTER(_Tensor4)] * 3 + [c_int, c_int, c_int, c_vp, c_vp]
    lib.ulysses_merge_output_head_chunk.restype = c_int
    lib.ulysses_merge_output_head_chunk.argtypes = [ctypes.POINTER(_Tensor4), c_int, c_int, c_int, c_vp, c_vp]
    lib.ulysses_pack_head_chunk_schedule.restype = c_int
    lib.ulysses_pack_head_chunk_schedule.argtypes = [ctypes.POINTER(_Tensor4)] * 3 + [
        c_int, c_int, ctypes.POINTER(c_int), ctypes.POINTER(c_int), ctypes.POINTER(c_vp), c_vp]
    lib.ulysses_merge_output_head_chunk_schedule.restype = c_int
    lib.ulysses_merge_output_head_chunk_schedule.argtypes = [ctypes.POINTER(ctypes.POINTER(_Tensor4)), c_int, c_int,
                                                            c_int, ctypes.POINTER(c_int), c_vp, c_vp]
    lib.qnre_forward_noalloc.restype = c_int
    lib.qnre_forward_noalloc.argtypes = [c_int, c_int, c_int, c_int, c_int, c_uint, c_int, c_int,
                                         c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, ctypes.POINTER(_Out), c_vp, c_vp]
    i32 = ctypes.c_int32
    lib.ulysses_scatter_heads.restype = c_int
    lib.ulysses_scatter_heads.argtypes = [c_vp, c_int, c_int, c_int, c_int, c_int, i32, c_vp, c_vp]
    lib.ulysses_gather_heads.restype = c_int
    lib.ulysses_gather_heads.argtypes = [c_vp, c_int, c_int, c_int, c_int, c_int, i32, c_vp, c_vp]
    lib.ulysses_pack_output_sequence_chunk.restype = c_int
    lib.ulysses_pack_output_sequence_chunk.argtypes = [ctypes.POINTER(_Tensor4), c_int, c_vp, c_vp]
    lib.ulysses_gather_output_head_chunk.restype = c_int
    lib.ulysses_gather_output_head_chunk.argtypes = [c_vp, c_int, c_int, c_int, c_int, c_int, i32, c_int, c_int,
                                                     c_vp, c_vp]
    lib.ulysses_scatter_qkv_head_chunk.restype = c_int
    lib.ulysses_scatter_qkv_head_chunk.argtypes = [ctypes.POINTER(_Tensor4)] * 3 + [c_int, c_int, c_int, c_vp, c_vp]
    lib.qnre_forward_publish.restype = c_int
    lib.qnre_forward_publish.argtypes = [c_vp, c_int, c_int, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp,
                                         ctypes.POINTER(_Out), c_vp, c_vp]
    lib.qnre_ready_target.restype = c_int
    lib.qnre_ready_target.argtypes = [c_vp, c_int, c_int, ctypes.POINTER(c_uint)]
    lib.qnre_wait_ready.restype = c_int
    lib.qnre_wait_ready.argtypes = [c_vp, c_vp, c_uint, ctypes.c_uint64, c_vp]
    lib.ulysses_sage2_workspace_bytes.restype = c_int
    lib.ulysses_sage2_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(ctypes.c_uint64)]
    lib.ulysses_sage2_scatter_qkv.restype = c_int
    lib.ulysses_sage2_scatter_qkv.argtypes = [ctypes.POINTER(_Tensor4)] * 3 + [c_int, c_int] + [c_vp] * 7 + \
        [ctypes.c_uint64, c_vp]
    _lib = lib
    return lib


def header_functions(path: str = HEADER) -> List[str]:
    """Names of the functions include/qnre.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                      text, flags=re.M)


def _check(status: int, where: str) -> None:
    if status != QNRE_OK:
        raise QnreError(status, where)


def _dtype_code(t) -> int:
    import torch
    codes = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
    if t.dtype not in codes:
        raise QnreError(2, f"dtype {t.dtype}")
    return codes[t.dtype]


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _tensor4(t) -> _Tensor4:
    if t.dim() != 4:
        raise QnreError(1, "expected a rank-4 view")
    d = _Tensor4()
    d.data = t.data_ptr()
    for i in range(4):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    d.dtype = _dtype_code(t)
    return d


class Plan:
    """qnre_plan_create / qnre_plan_destroy."""

    def __init__(self, hidden: int, num_heads: int, P: int, layout: str = "bshd",
                 max_tokens: int = 1, rope_style: str = "rotate_half", head_dim: int = HEAD_DIM,
                 flags: int = 0):
        lib = load_library()
        self._handle = ctypes.c_void_p()
        self.hidden, self.num_heads, self.P = hidden, num_heads, P
        self.layout, self.rope_style, self.max_tokens, self.flags = layout, rope_style, max_tokens, flags
        _check(lib.qnre_plan_create(ctypes.byref(self._handle), hidden, num_heads, head_dim, P,
                                    LAYOUTS.get(layout, -1), max_tokens, ROPE_STYLES.get(rope_style, -1),
                                    flags), "qnre_plan_create")

    @property
    def handle(self):
        return self._handle

    def destroy(self) -> None:
        if self._handle:
            _check(load_library().qnre_plan_destroy(self._handle), "qnre_plan_destroy")
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            if self._handle:
                load_library().qnre_plan_destroy(self._handle)
        except Exception:
            pass

    def reserve_sms(self, sms: int) -> None:
        """qnre_plan_reserve_sms: leave `sms` SMs free of the fused kernel (0 = use all)."""
        _check(load_library().qnre_plan_reserve_sms(self._handle, sms), "qnre_plan_reserve_sms")

    def describe(self, B: int, S_local: int) -> Dict[str, int]:
        """qnre_plan_describe: how a forward of (B, S_local) runs (clusters, SMs, work list)."""
        info = _PlanInfo()
        _check(load_library().qnre_plan_describe(self._handle, B, S_local, ctypes.byref(info)),
               "qnre_plan_describe")
        return {name: getattr(info, name) for name, _ in _PlanInfo._fields_}

    def device_status(self, clear: bool = True, stream=None) -> int:
        bits = ctypes.c_uint(0)
        st = load_library().qnre_plan_device_status(self._handle, _stream_ptr(stream), ctypes.byref(bits),
                                                    1 if clear else 0)
        if st not in (QNRE_OK, 7):
            raise QnreError(st, "qnre_plan_device_status")
        return bits.value


def debug_bounds(reset: bool = True) -> int:
    """Accesses the debug build's layout and Sage2 kernels skipped (qnre_debug_bounds);
    raises QnreError(QNRE_ERR_UNSUPPORTED) on the release build."""
    n = ctypes.c_ulonglong(0)
    st = load_library().qnre_debug_bounds(ctypes.byref(n), 1 if reset else 0)
    if st != QNRE_OK:
        raise QnreError(st, "qnre_debug_bounds")
    return n.value


def qnre_forward(plan: Plan, x, w_qkv, q_norm_w, k_norm_w, cos_sin, positions, out: Dict[str, object],
                 stream=None) -> None:
    """x: bf16 [P, B, S_local, hidden]; out: {"q","k","v"} (bshd) or {"fused"} (fused)."""
    if x.dim() != 4 or x.shape[0] != plan.P:
        raise QnreError(1, "qnre_forward: x must be [P, B, S_local, hidden]")
    o = _Out(_ptr(out.get("q")), _ptr(out.get("k")), _ptr(out.get("v")), _ptr(out.get("fused")))
    _check(load_library().qnre_forward(plan.handle, x.shape[1], x.shape[2], x.data_ptr(), w_qkv.data_ptr(),
                                       q_norm_w.data_ptr(), k_norm_w.data_ptr(), cos_sin.data_ptr(),
                                       cos_sin.shape[0], _ptr(positions), ctypes.byref(o),
                                       _stream_ptr(stream)), "qnre_forward")


def ulysses_pack_head_chunk(q, k, v, world_size: int, head_offset: int, head_count: int, out,
                            stream=None):
    """Pack one head band of strided q/k/v [B, S, H, D] into contiguous out [B, S, W*cnt, 3D]."""
    tq, tk, tv = _tensor4(q), _tensor4(k), _tensor4(v)
    _check(load_library().ulysses_pack_head_chunk(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                                  world_size, head_offset, head_count, out.data_ptr(),
                                                  _stream_ptr(stream)), "ulysses_pack_head_chunk")
    return out


def ulysses_merge_output_head_chunk(received, world_size: int, local_heads: int, head_offset: int, out,
                                    stream=None):
    """Merge received [B, S, W*cnt, D] into band head_offset of contiguous out [B, S, W*L, D]."""
    tr = _tensor4(received)
    _check(load_library().ulysses_merge_output_head_chunk(ctypes.byref(tr), world_size, local_heads,
                                                          head_offset, out.data_ptr(), _stream_ptr(stream)),
           "ulysses_merge_output_head_chunk")
    return out


def ulysses_pack_head_chunk_schedule(q, k, v, world_size: int, schedule, outs, stream=None):
    """Every (head_offset, head_count) chunk of `schedule` packed into outs[i] in one launch."""
    n = len(schedule)
    tq, tk, tv = _tensor4(q), _tensor4(k), _tensor4(v)
    offs = (ctypes.c_int * n)(*[int(o) for o, _ in schedule])
    cnts = (ctypes.c_int * n)(*[int(c) for _, c in schedule])
    ptrs = (ctypes.c_void_p * n)(*[_contig(o, "pack_head_chunk_schedule") for o in outs])
    _check(load_library().ulysses_pack_head_chunk_schedule(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                                           world_size, n, offs, cnts, ptrs, _stream_ptr(stream)),
           "ulysses_pack_head_chunk_schedule")
    return outs


def ulysses_merge_output_head_chunk_schedule(received, world_size: int, local_heads: int, head_offsets, out,
                                             stream=None):
    """Every received[i] merged at band head_offsets[i] of `out` in one launch."""
    n = len(received)
    views = [_tensor4(r) for r in received]
    arr = (ctypes.POINTER(_Tensor4) * n)(*[ctypes.pointer(t) for t in views])
    offs = (ctypes.c_int * n)(*[int(o) for o in head_offsets])
    _check(load_library().ulysses_merge_output_head_chunk_schedule(arr, world_size, local_heads, n, offs,
                                                                   _contig(out, "merge_output_head_chunk_schedule"),
                                                                   _stream_ptr(stream)),
           "ulysses_merge_output_head_chunk_schedule")
    return out


def qnre_forward_publish(plan: Plan, x, w_qkv, q_norm_w, k_norm_w, cos_sin, positions, out: Dict[str, object],
                         ready, stream=None) -> None:
    """qnre_forward that also publishes per-destination readiness counts into ready (int32 CUDA [P])."""
    if x.dim() != 4 or x.shape[0] != plan.P:
        raise QnreError(1, "qnre_forward_publish: x must be [P, B, S_local, hidden]")
    o = _Out(_ptr(out.get("q")), _ptr(out.get("k")), _ptr(out.get("v")), _ptr(out.get("fused")))
    _check(load_library().qnre_forward_publish(plan.handle, x.shape[1], x.shape[2], x.data_ptr(), w_qkv.data_ptr(),
                                               q_norm_w.data_ptr(), k_norm_w.data_ptr(), cos_sin.data_ptr(),
                                               cos_sin.shape[0], _ptr(positions), ctypes.byref(o), ready.data_ptr(),
                                               _stream_ptr(stream)), "qnre_forward_publish")


def qnre_ready_target(plan: Plan, B: int, S_local: int) -> int:
    t = ctypes.c_uint(0)
    _check(load_library().qnre_ready_target(plan.handle, B, S_local, ctypes.byref(t)), "qnre_ready_target")
    return t.value


def qnre_wait_ready(plan: Plan, ready, target: int, timeout_ns: int, stream=None) -> None:
    """Enqueue the bounded one-CTA wait for every ready[r] >= target; expiry sets DEVICE_READY_TIMEOUT."""
    _check(load_library().qnre_wait_ready(plan.handle, ready.data_ptr(), target, timeout_ns, _stream_ptr(stream)),
           "qnre_wait_ready")


def qnre_forward_noalloc(hidden: int, num_heads: int, P: int, x, w_qkv, q_norm_w, k_norm_w, cos_sin, positions,
                         out: Dict[str, object], layout: str = "bshd", rope_style: str = "rotate_half",
                         flags: int = 0, device_status=None, stream=None) -> None:
    """qnre_forward without a plan: for callers that cannot allocate device memory when they
    project.  device_status: optional int32 CUDA tensor of one element that receives the
    call's QNRE_DEVICE_* bits."""
    if x.dim() != 4 or x.shape[0] != P:
        raise QnreError(1, "qnre_forward_noalloc: x must be [P, B, S_local, hidden]")
    o = _Out(_ptr(out.get("q")), _ptr(out.get("k")), _ptr(out.get("v")), _ptr(out.get("fused")))
    _check(load_library().qnre_forward_noalloc(hidden, num_heads, P, LAYOUTS.get(layout, -1),
                                               ROPE_STYLES.get(rope_style, -1), flags, x.shape[1], x.shape[2],
                                               x.data_ptr(), w_qkv.data_ptr(), q_norm_w.data_ptr(),
                                               k_norm_w.data_ptr(), cos_sin.data_ptr(), cos_sin.shape[0],
                                               _ptr(positions), ctypes.byref(o), _ptr(device_status),
                                               _stream_ptr(stream)), "qnre_forward_noalloc")


def _contig(t, where: str):
    if not t.is_contiguous():
        raise QnreError(1, f"{where}: tensor must be contiguous")
    return t.data_ptr()


def ulysses_scatter_heads(x, out, stream=None):
    """x [P, B, S_local, H, D] -> out [P, B, P*S_local, H/P, D] (both contiguous)."""
    P, B, S, H, D = x.shape
    _check(load_library().ulysses_scatter_heads(_contig(x, "scatter_heads"), P, B, S, H, D, _dtype_code(x),
                                                _contig(out, "scatter_heads"), _stream_ptr(stream)),
           "ulysses_scatter_heads")
    return out


def ulysses_gather_heads(y, out, stream=None):
    """y [P, B, S_global, H_local, D] -> out [P, B, S_global/P, P*H_local, D] (both contiguous)."""
    P, B, S_g, H_l, D = y.shape
    _check(load_library().ulysses_gather_heads(_contig(y, "gather_heads"), P, B, S_g, H_l, D, _dtype_code(y),
                                               _contig(out, "gather_heads"), _stream_ptr(stream)),
           "ulysses_gather_heads")
    return out


def ulysses_pack_output_sequence_chunk(x, world_size: int, out, stream=None):
    """x view [B, S_global, head_count, D] -> out [world_size, B, S_global/world_size, head_count, D]."""
    tx = _tensor4(x)
    _check(load_library().ulysses_pack_output_sequence_chunk(ctypes.byref(tx), world_size,
                                                             _contig(out, "pack_output_sequence_chunk"),
                                                             _stream_ptr(stream)),
           "ulysses_pack_output_sequence_chunk")
    return out


def ulysses_gather_output_head_chunk(x, local_heads: int, head_offset: int, out, stream=None):
    """x [P, B, S_global, head_count, D] -> band head_offset of out [P, B, S_global/P, P*local_heads, D]."""
    P, B, S_g, cnt, D = x.shape
    _check(load_library().ulysses_gather_output_head_chunk(_contig(x, "gather_output_head_chunk"), P, B, S_g, cnt, D,
                                                           _dtype_code(x), local_heads, head_offset,
                                                           _contig(out, "gather_output_head_chunk"),
                                                           _stream_ptr(stream)),
           "ulysses_gather_output_head_chunk")
    return out


def ulysses_scatter_qkv_head_chunk(q, k, v, P: int, head_offset: int, head_count: int, out, stream=None):
    """q/k/v views [P*B, S_local, H, D] -> out [P, B, P*S_local, head_count, 3*D] (contiguous)."""
    tq, tk, tv = _tensor4(q), _tensor4(k), _tensor4(v)
    _check(load_library().ulysses_scatter_qkv_head_chunk(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), P,
                                                         head_offset, head_count,
                                                         _contig(out, "scatter_qkv_head_chunk"),
                                                         _stream_ptr(stream)),
           "ulysses_scatter_qkv_head_chunk")
    return out


def alloc_outputs(plan: Plan, B: int, S_local: int, device="cuda") -> Dict[str, object]:
    """Output buffers for qnre_forward (uninitialised bf16)."""
    import torch
    H_local = plan.num_heads // plan.P
    S_g = plan.P * S_local
    if plan.layout == "bshd":
        return {g: torch.empty((plan.P, B, S_g, H_local, HEAD_DIM), dtype=torch.bfloat16, device=device)
                for g in "qkv"}
    return {"fused": torch.empty((plan.P, B, S_g, H_local, 3 * HEAD_DIM), dtype=torch.bfloat16, device=device)}


def ulysses_sage2_workspace_bytes(P: int, B: int, L: int, H: int, D: int) -> int:
    """Scratch bytes ulysses_sage2_scatter_qkv needs for these sizes."""
    n = ctypes.c_uint64()
    _check(load_library().ulysses_sage2_workspace_bytes(P, B, L, H, D, ctypes.byref(n)),
           "ulysses_sage2_workspace_bytes")
    return n.value


def sage2_outputs(P: int, B: int, L: int, H: int, D: int, used_sequence: int, device="cuda") -> Dict[str, object]:
    """Output buffers (uninitialised) and the workspace for ulysses_sage2_scatter_qkv."""
    import torch
    S, H_l = P * L, H // P
    S_pad = -(-S // 64) * 64
    U = used_sequence
    ws = ulysses_sage2_workspace_bytes(P, B, L, H, D)
    return {"q": torch.empty((P, B, S, H_l, D), dtype=torch.int8, device=device),
            "k": torch.empty((P, B, S, H_l, D), dtype=torch.int8, device=device),
            "v": torch.empty((P, B, D, H_l, S_pad), dtype=torch.uint8, device=device),
            "q_scale": torch.empty((P, B, H_l, -(-U // 32)), dtype=torch.float32, device=device),
            "k_scale": torch.empty((P, B, H_l, -(-U // 64)), dtype=torch.float32, device=device),
            "v_scale": torch.empty((P, B, H_l, D), dtype=torch.float32, device=device),
            "workspace": torch.empty((ws,), dtype=torch.uint8, device=device)}


def ulysses_sage2_scatter_qkv(q, k, v, P: int, used_sequence: int, out: Dict[str, object], stream=None):
    """q/k/v views [P*B, L, H, D] (bf16 or fp16) -> the Sage2 codes and scales of every
    destination rank in `out` (see sage2_outputs)."""
    tq, tk, tv = _tensor4(q), _tensor4(k), _tensor4(v)
    names = ("q", "k", "v", "q_scale", "k_scale", "v_scale")
    ptrs = [_contig(out[n], "sage2_scatter_qkv") for n in names]
    ws = out["workspace"]
    _check(load_library().ulysses_sage2_scatter_qkv(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), P,
                                                    used_sequence, *ptrs, _contig(ws, "sage2_scatter_qkv"),
                                                    ws.numel() * ws.element_size(), _stream_ptr(stream)),
           "ulysses_sage2_scatter_qkv")
    return out
