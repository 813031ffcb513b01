"""ctypes binding of libbl_attn.so (argument marshalling only).

Every function takes torch CUDA tensors, checks dtype/shape/contiguity and
passes raw device pointers plus the current CUDA stream to the C ABI
declared in ``include/bl_attn.h``.  There is no fallback: if the library is
missing or a call fails, a RuntimeError is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbl_attn.so")

BL_STATUS = {0: "BL_OK", 1: "BL_ERR_INVALID_ARG", 2: "BL_ERR_UNSUPPORTED", 3: "BL_ERR_CUDA",
             4: "BL_ERR_WORKSPACE", 5: "BL_ERR_CORRUPT_LISTS", 6: "BL_ERR_TIMEOUT"}

# Every symbol include/bl_attn.h declares (checked by the CPU test suite).
EXPORTS = ("bl_tile_stats_elems", "bl_lists_elems", "bl_bwd_workspace_bytes", "bl_attn_fwd",
           "bl_mask_from_stats", "bl_fwd_workspace_bytes", "bl_attn_fwd_tile_weights",
           "bl_mask_from_tile_weights", "bl_attn_bwd", "bl_bwd_check_status", "bl_status_string",
           "bl_attn_bwd_noalloc", "bl_bwd_noalloc_check_status", "bl_lse_combine", "bl_grad_error", "bl_varlen_layout",
           "bl_attn_fwd_varlen", "bl_mask_from_stats_varlen", "bl_fwd_workspace_bytes_varlen",
           "bl_attn_fwd_tile_weights_varlen", "bl_mask_from_tile_weights_varlen",
           "bl_attn_bwd_varlen",
           "bl_varlen_bwd_check_status", "bl_set_wait_limit")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("n", ctypes.c_int), ("H", ctypes.c_int),
                ("Hk", ctypes.c_int), ("d", ctypes.c_int), ("block_q", ctypes.c_int),
                ("block_k", ctypes.c_int), ("causal", ctypes.c_int), ("window", ctypes.c_int),
                ("q_strides", ctypes.c_int64 * 4), ("k_strides", ctypes.c_int64 * 4),
                ("v_strides", ctypes.c_int64 * 4), ("o_strides", ctypes.c_int64 * 4)]

    def strides_of(self, role):
        """Element strides a tensor of this role (q, k, v, o) must have, or None
        when the shape's are all zero (a contiguous tensor)."""
        st = tuple(getattr(self, role + "_strides"))
        return st if any(st) else None


class Lists(ctypes.Structure):
    _fields_ = [("mask", ctypes.c_void_p), ("kv_idx", ctypes.c_void_p),
                ("kv_cnt", ctypes.c_void_p), ("q_idx", ctypes.c_void_p),
                ("q_cnt", ctypes.c_void_p), ("nan_count", ctypes.c_void_p)]


class VarlenStruct(ctypes.Structure):
    _fields_ = [("nseq", ctypes.c_int), ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)),
                ("H", ctypes.c_int), ("Hk", ctypes.c_int), ("d", ctypes.c_int),
                ("block_q", ctypes.c_int), ("block_k", ctypes.c_int), ("causal", ctypes.c_int),
                ("window", ctypes.c_int), ("streams", ctypes.c_int)]


class VarlenSizes(ctypes.Structure):
    _fields_ = [("total", ctypes.c_size_t), ("lse", ctypes.c_size_t),
                ("tile_stats", ctypes.c_size_t), ("mask", ctypes.c_size_t),
                ("kv_cnt", ctypes.c_size_t), ("q_idx", ctypes.c_size_t),
                ("q_cnt", ctypes.c_size_t), ("bwd_workspace_bytes", ctypes.c_size_t),
                ("groups", ctypes.c_int)]


class BLError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} failed: {BL_STATUS.get(code, code)}")


_lib = None


def load():
    """Load libbl_attn.so once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m block_sparse_attention_fwd_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    P, S, F, D, Z = ctypes.c_void_p, ctypes.POINTER(Shape), ctypes.c_float, ctypes.c_double, ctypes.c_size_t
    lib.bl_tile_stats_elems.argtypes = [S]
    lib.bl_tile_stats_elems.restype = Z
    lib.bl_lists_elems.argtypes = [S, ctypes.POINTER(ctypes.c_size_t)]
    lib.bl_lists_elems.restype = Z
    lib.bl_bwd_workspace_bytes.argtypes = [S]
    lib.bl_bwd_workspace_bytes.restype = Z
    lib.bl_attn_fwd.argtypes = [S, P, P, P, F, P, P, P, P]
    lib.bl_attn_fwd.restype = ctypes.c_int
    lib.bl_mask_from_stats.argtypes = [S, P, P, D, ctypes.POINTER(Lists), P]
    lib.bl_mask_from_stats.restype = ctypes.c_int
    lib.bl_fwd_workspace_bytes.argtypes = [S]
    lib.bl_fwd_workspace_bytes.restype = Z
    lib.bl_attn_fwd_tile_weights.argtypes = [S, P, P, P, F, P, P, P, P, P, Z, P]
    lib.bl_attn_fwd_tile_weights.restype = ctypes.c_int
    lib.bl_mask_from_tile_weights.argtypes = [S, P, D, ctypes.POINTER(Lists), P]
    lib.bl_mask_from_tile_weights.restype = ctypes.c_int
    lib.bl_attn_bwd.argtypes = [S, P, P, P, P, P, P, F, ctypes.POINTER(Lists), P, P, P, P, Z, P]
    lib.bl_attn_bwd.restype = ctypes.c_int
    lib.bl_attn_bwd_noalloc.argtypes = [S, P, P, P, P, P, P, F, ctypes.POINTER(Lists), P, P, P, P]
    lib.bl_attn_bwd_noalloc.restype = ctypes.c_int
    lib.bl_bwd_noalloc_check_status.argtypes = [S, P]
    lib.bl_bwd_noalloc_check_status.restype = ctypes.c_int
    lib.bl_lse_combine.argtypes = [ctypes.c_int] * 5 + [P, P, P, P, P]
    lib.bl_lse_combine.restype = ctypes.c_int
    lib.bl_grad_error.argtypes = [P, P, Z, P, P]
    lib.bl_grad_error.restype = ctypes.c_int
    lib.bl_bwd_check_status.argtypes = [S, P, P]
    lib.bl_bwd_check_status.restype = ctypes.c_int
    V = ctypes.POINTER(VarlenStruct)
    lib.bl_varlen_layout.argtypes = [V, ctypes.POINTER(VarlenSizes)]
    lib.bl_varlen_layout.restype = ctypes.c_int
    lib.bl_attn_fwd_varlen.argtypes = [V, P, P, P, F, P, P, P, P]
    lib.bl_attn_fwd_varlen.restype = ctypes.c_int
    lib.bl_mask_from_stats_varlen.argtypes = [V, P, P, D, ctypes.POINTER(Lists), P]
    lib.bl_mask_from_stats_varlen.restype = ctypes.c_int
    lib.bl_fwd_workspace_bytes_varlen.argtypes = [V]
    lib.bl_fwd_workspace_bytes_varlen.restype = ctypes.c_size_t
    lib.bl_attn_fwd_tile_weights_varlen.argtypes = [V, P, P, P, F, P, P, P, P, P, Z, P]
    lib.bl_attn_fwd_tile_weights_varlen.restype = ctypes.c_int
    lib.bl_mask_from_tile_weights_varlen.argtypes = [V, P, D, ctypes.POINTER(Lists), P]
    lib.bl_mask_from_tile_weights_varlen.restype = ctypes.c_int
    lib.bl_attn_bwd_varlen.argtypes = [V, P, P, P, P, P, P, F, ctypes.POINTER(Lists), P, P, P,
                                       P, Z, P]
    lib.bl_attn_bwd_varlen.restype = ctypes.c_int
    lib.bl_varlen_bwd_check_status.argtypes = [V, P, P]
    lib.bl_varlen_bwd_check_status.restype = ctypes.c_int
    lib.bl_set_wait_limit.argtypes = [D]
    lib.bl_set_wait_limit.restype = D
    lib.bl_status_string.argtypes = [ctypes.c_int]
    lib.bl_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(fn, code):
    if code != 0:
        raise BLError(fn, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, dtype, shape, name, strides=None):
    """Checks a tensor argument.  strides: the element strides a BSHD view must
    have (from the bl_shape); None means contiguous."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if strides is None:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    elif any(sz > 1 and a != b for sz, a, b in zip(t.shape, t.stride(), strides)) or \
            t.stride()[-1] != 1:
        raise ValueError(f"{name} has strides {tuple(t.stride())}, the shape says {strides}")


def make_shape(B, n, H, Hk, d, block_q, block_k, causal=0, window=0) -> Shape:
    """A shape for contiguous BSHD tensors (all strides zero)."""
    return Shape(B, n, H, Hk, d, block_q, block_k, int(causal), int(window))


def with_strides(shape: Shape, q=None, k=None, v=None, o=None) -> Shape:
    """A copy of `shape` whose strides are those of the given BSHD views (q for
    q/g_q, k for k/g_k, v for v/g_v, o for o/g_o); roles not given stay as they
    are.  Every view must have a contiguous last dim."""
    out = Shape.from_buffer_copy(shape)
    for role, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if t is None:
            continue
        st = tuple(int(x) for x in t.stride())
        if len(st) != 4 or st[3] != 1:
            raise ValueError(f"{role}: a BSHD view with a contiguous last dim is needed")
        arr = getattr(out, role + "_strides")
        for i, x in enumerate(st):
            arr[i] = x
    return out


def tiles(shape: Shape):
    T_r = -(-shape.n // shape.block_q)
    T_c = -(-shape.n // shape.block_k)
    return T_r, T_c


def tile_stats_elems(shape: Shape) -> int:
    return int(load().bl_tile_stats_elems(ctypes.byref(shape)))


def lists_elems(shape: Shape):
    """(element counts of mask, kv_idx, kv_cnt, q_idx, q_cnt, total bytes)."""
    out = (ctypes.c_size_t * 5)()
    total = int(load().bl_lists_elems(ctypes.byref(shape), out))
    return tuple(int(x) for x in out) + (total,)


def bwd_workspace_bytes(shape: Shape) -> int:
    return int(load().bl_bwd_workspace_bytes(ctypes.byref(shape)))


def attn_fwd(shape, q, k, v, scale, o, lse, tile_stats=None):
    B, n, H, Hk, d = shape.B, shape.n, shape.H, shape.Hk, shape.d
    _need(q, torch.bfloat16, (B, n, H, d), "q", shape.strides_of("q"))
    _need(k, torch.bfloat16, (B, n, Hk, d), "k", shape.strides_of("k"))
    _need(v, torch.bfloat16, (B, n, Hk, d), "v", shape.strides_of("v"))
    _need(o, torch.bfloat16, (B, n, H, d), "o", shape.strides_of("o"))
    _need(lse, torch.float32, (B, H, n), "lse")
    if tile_stats is not None:
        T_r, T_c = tiles(shape)
        _need(tile_stats, torch.float32, (B, H, T_c, T_r * shape.block_q), "tile_stats")
    code = load().bl_attn_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), float(scale),
                              _ptr(o), _ptr(lse), _ptr(tile_stats), _stream(q.device))
    _check("bl_attn_fwd", code)


def fwd_tile_weights_supported(shape: Shape) -> bool:
    """Whether bl_attn_fwd_tile_weights takes this shape (the header's rule:
    tiles of 64 or 128, head dim 64 or 128, T_c <= 2048)."""
    return (shape.block_q in (64, 128) and shape.block_k in (64, 128) and shape.d in (64, 128)
            and tiles(shape)[1] <= 2048)


def fwd_workspace_bytes(shape: Shape) -> int:
    """Scratch of attn_fwd_tile_weights without a statistics output (current device)."""
    return int(load().bl_fwd_workspace_bytes(ctypes.byref(shape)))


def attn_fwd_tile_weights(shape, q, k, v, scale, o, lse, tile_logw, tile_stats=None,
                          workspace=None):
    """bl_attn_fwd_tile_weights: the forward that also reduces the tile weights
    tile_logw [B,H,T_r,T_c] fp32; without tile_stats the statistics rows live
    only in `workspace` (uint8, at least fwd_workspace_bytes)."""
    B, n, H, Hk, d = shape.B, shape.n, shape.H, shape.Hk, shape.d
    T_r, T_c = tiles(shape)
    _need(q, torch.bfloat16, (B, n, H, d), "q", shape.strides_of("q"))
    _need(k, torch.bfloat16, (B, n, Hk, d), "k", shape.strides_of("k"))
    _need(v, torch.bfloat16, (B, n, Hk, d), "v", shape.strides_of("v"))
    _need(o, torch.bfloat16, (B, n, H, d), "o", shape.strides_of("o"))
    _need(lse, torch.float32, (B, H, n), "lse")
    _need(tile_logw, torch.float32, (B, H, T_r, T_c), "tile_logw")
    if tile_stats is not None:
        _need(tile_stats, torch.float32, (B, H, T_c, T_r * shape.block_q), "tile_stats")
    nbytes = 0
    if workspace is not None:
        if workspace.dtype != torch.uint8 or not workspace.is_cuda:
            raise TypeError("workspace must be a CUDA uint8 tensor")
        nbytes = workspace.numel()
    code = load().bl_attn_fwd_tile_weights(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v),
                                           float(scale), _ptr(o), _ptr(lse), _ptr(tile_stats),
                                           _ptr(tile_logw), _ptr(workspace), nbytes,
                                           _stream(q.device))
    _check("bl_attn_fwd_tile_weights", code)


def mask_from_tile_weights(shape, tile_logw, negl_prob, lists):
    B, H = shape.B, shape.H
    T_r, T_c = tiles(shape)
    _need(tile_logw, torch.float32, (B, H, T_r, T_c), "tile_logw")
    _need(lists["mask"], torch.uint8, (B, H, T_r, T_c), "mask")
    _need(lists["kv_idx"], torch.int32, (B, H, T_r, T_c), "kv_idx")
    _need(lists["kv_cnt"], torch.int32, (B, H, T_r), "kv_cnt")
    _need(lists["q_idx"], torch.int32, (B, H, T_c, T_r), "q_idx")
    _need(lists["q_cnt"], torch.int32, (B, H, T_c), "q_cnt")
    ls = _lists_struct(lists)
    code = load().bl_mask_from_tile_weights(ctypes.byref(shape), _ptr(tile_logw),
                                            float(negl_prob), ctypes.byref(ls),
                                            _stream(tile_logw.device))
    _check("bl_mask_from_tile_weights", code)


def alloc_lists(shape: Shape, device) -> dict:
    T_r, T_c = tiles(shape)
    B, H = shape.B, shape.H
    return {
        "mask": torch.empty((B, H, T_r, T_c), dtype=torch.uint8, device=device),
        "kv_idx": torch.empty((B, H, T_r, T_c), dtype=torch.int32, device=device),
        "kv_cnt": torch.empty((B, H, T_r), dtype=torch.int32, device=device),
        "q_idx": torch.empty((B, H, T_c, T_r), dtype=torch.int32, device=device),
        "q_cnt": torch.empty((B, H, T_c), dtype=torch.int32, device=device),
        "nan_count": torch.zeros((1,), dtype=torch.int32, device=device),
    }


def _lists_struct(lists):
    return Lists(_ptr(lists["mask"]), _ptr(lists["kv_idx"]), _ptr(lists["kv_cnt"]),
                 _ptr(lists["q_idx"]), _ptr(lists["q_cnt"]), _ptr(lists.get("nan_count")))


def mask_from_stats(shape, tile_stats, lse, negl_prob, lists):
    B, H, n = shape.B, shape.H, shape.n
    T_r, T_c = tiles(shape)
    _need(tile_stats, torch.float32, (B, H, T_c, T_r * shape.block_q), "tile_stats")
    _need(lse, torch.float32, (B, H, n), "lse")
    _need(lists["mask"], torch.uint8, (B, H, T_r, T_c), "mask")
    _need(lists["kv_idx"], torch.int32, (B, H, T_r, T_c), "kv_idx")
    _need(lists["kv_cnt"], torch.int32, (B, H, T_r), "kv_cnt")
    _need(lists["q_idx"], torch.int32, (B, H, T_c, T_r), "q_idx")
    _need(lists["q_cnt"], torch.int32, (B, H, T_c), "q_cnt")
    ls = _lists_struct(lists)
    code = load().bl_mask_from_stats(ctypes.byref(shape), _ptr(tile_stats), _ptr(lse),
                                     float(negl_prob), ctypes.byref(ls), _stream(lse.device))
    _check("bl_mask_from_stats", code)


def _bwd_tensors(shape, q, k, v, o, g_o, g_q, g_k, g_v):
    B, n, H, Hk, d = shape.B, shape.n, shape.H, shape.Hk, shape.d
    for t, nm, sh, role in ((q, "q", (B, n, H, d), "q"), (k, "k", (B, n, Hk, d), "k"),
                            (v, "v", (B, n, Hk, d), "v"), (o, "o", (B, n, H, d), "o"),
                            (g_o, "g_o", (B, n, H, d), "o"), (g_q, "g_q", (B, n, H, d), "q"),
                            (g_k, "g_k", (B, n, Hk, d), "k"), (g_v, "g_v", (B, n, Hk, d), "v")):
        _need(t, torch.bfloat16, sh, nm, shape.strides_of(role))


def attn_bwd(shape, q, k, v, o, g_o, lse, scale, lists, g_q, g_k, g_v, workspace):
    B, n, H, Hk, d = shape.B, shape.n, shape.H, shape.Hk, shape.d
    _bwd_tensors(shape, q, k, v, o, g_o, g_q, g_k, g_v)
    _need(lse, torch.float32, (B, H, n), "lse")
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA uint8 tensor")
    ls = None
    if lists is not None:
        T_r, T_c = tiles(shape)
        _need(lists["q_idx"], torch.int32, (B, H, T_c, T_r), "q_idx")
        _need(lists["q_cnt"], torch.int32, (B, H, T_c), "q_cnt")
        ls = _lists_struct(lists)
    code = load().bl_attn_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(g_o),
                              _ptr(lse), float(scale),
                              ctypes.byref(ls) if ls is not None else None,
                              _ptr(g_q), _ptr(g_k), _ptr(g_v), _ptr(workspace),
                              workspace.numel(), _stream(q.device))
    _check("bl_attn_bwd", code)


def bwd_check_status(shape, workspace) -> int:
    return int(load().bl_bwd_check_status(ctypes.byref(shape), _ptr(workspace),
                                          _stream(workspace.device)))


def attn_bwd_noalloc(shape, q, k, v, o, g_o, lse, scale, lists, g_q, g_k, g_v):
    """bl_attn_bwd_noalloc: the backward with the library's fixed device scratch
    instead of a workspace (for callers that cannot allocate device memory)."""
    B, n, H, Hk, d = shape.B, shape.n, shape.H, shape.Hk, shape.d
    _bwd_tensors(shape, q, k, v, o, g_o, g_q, g_k, g_v)
    _need(lse, torch.float32, (B, H, n), "lse")
    ls = _lists_struct(lists) if lists is not None else None
    code = load().bl_attn_bwd_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                      _ptr(g_o), _ptr(lse), float(scale),
                                      ctypes.byref(ls) if ls is not None else None,
                                      _ptr(g_q), _ptr(g_k), _ptr(g_v), _stream(q.device))
    _check("bl_attn_bwd_noalloc", code)


def set_wait_limit(seconds: float) -> float:
    """bl_set_wait_limit: the device-side wait limit for later launches (seconds
    in [0, 2); anything else restores 2 s).  Returns the previous limit."""
    return float(load().bl_set_wait_limit(float(seconds)))


def bwd_noalloc_check_status(shape, device=None) -> int:
    """bl_bwd_noalloc_check_status: the status word of the last no-alloc backward."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    return int(load().bl_bwd_noalloc_check_status(ctypes.byref(shape), _stream(dev)))


def lse_combine(o_parts, lse_parts, o, lse):
    """bl_lse_combine: o_parts [P,B,n,H,d] bf16, lse_parts [P,B,H,n] fp32 ->
    o [B,n,H,d] bf16, lse [B,H,n] fp32."""
    P, B, n, H, d = o_parts.shape
    _need(o_parts, torch.bfloat16, (P, B, n, H, d), "o_parts")
    _need(lse_parts, torch.float32, (P, B, H, n), "lse_parts")
    _need(o, torch.bfloat16, (B, n, H, d), "o")
    _need(lse, torch.float32, (B, H, n), "lse")
    code = load().bl_lse_combine(P, B, n, H, d, _ptr(o_parts), _ptr(lse_parts), _ptr(o),
                                 _ptr(lse), _stream(o.device))
    _check("bl_lse_combine", code)


def grad_error(a, b, out=None):
    """bl_grad_error: fp64 sums of (a-b)^2, b^2, a*b, a^2 over two bf16 tensors of
    equal size (b the reference); returns (rel_l2, cos) as Python floats."""
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16 or a.numel() != b.numel():
        raise ValueError("a and b must be bf16 tensors of the same size")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("a and b must be contiguous")
    if out is None:
        out = torch.empty(4, dtype=torch.float64, device=a.device)
    code = load().bl_grad_error(_ptr(a), _ptr(b), a.numel(), _ptr(out), _stream(a.device))
    _check("bl_grad_error", code)
    d2, b2, ab, a2 = out.tolist()
    rel = (d2 / b2) ** 0.5 if b2 > 0 else (0.0 if d2 == 0 else float("inf"))
    den = (b2 * a2) ** 0.5
    cos = ab / den if den > 0 else (1.0 if d2 == 0 else 0.0)
    return rel, cos


# --- packed variable-length batches ------------------------------------------

class Varlen:
    """A packed batch description for the bl_*_varlen calls.  Holds the host
    copy of cu_seqlens (nseq + 1 int32 offsets) that the C struct points at,
    and the element counts bl_varlen_layout reports."""

    def __init__(self, cu_seqlens, H, Hk, d, block_q=128, block_k=128, causal=0, window=0,
                 streams=0):
        cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist")
                               else cu_seqlens)]
        self.cu_seqlens = cu
        self._cu = (ctypes.c_int32 * len(cu))(*cu)
        self.struct = VarlenStruct(len(cu) - 1, self._cu, H, Hk, d, block_q, block_k,
                                   int(causal), int(window), int(streams))
        self.H, self.Hk, self.d = H, Hk, d
        self.block_q, self.block_k = block_q, block_k
        self.causal, self.window = int(causal), int(window)
        sz = VarlenSizes()
        _check("bl_varlen_layout", load().bl_varlen_layout(ctypes.byref(self.struct),
                                                           ctypes.byref(sz)))
        self.sizes = {f: getattr(sz, f) for f, _ in VarlenSizes._fields_}

    @property
    def total(self):
        return self.sizes["total"]

    def seq_shape(self, s):
        """The fixed-length shape (B = 1) of sequence s alone."""
        n = self.cu_seqlens[s + 1] - self.cu_seqlens[s]
        return make_shape(1, n, self.H, self.Hk, self.d, self.block_q, self.block_k,
                          self.causal, self.window)


def alloc_varlen_lists(vl: Varlen, device) -> dict:
    z = vl.sizes
    return {
        "mask": torch.empty(z["mask"], dtype=torch.uint8, device=device),
        "kv_idx": torch.empty(z["mask"], dtype=torch.int32, device=device),
        "kv_cnt": torch.empty(z["kv_cnt"], dtype=torch.int32, device=device),
        "q_idx": torch.empty(z["q_idx"], dtype=torch.int32, device=device),
        "q_cnt": torch.empty(z["q_cnt"], dtype=torch.int32, device=device),
        "nan_count": torch.zeros((1,), dtype=torch.int32, device=device),
    }


def attn_fwd_varlen(vl: Varlen, q, k, v, scale, o, lse, tile_stats=None):
    T, H, Hk, d = vl.total, vl.H, vl.Hk, vl.d
    _need(q, torch.bfloat16, (T, H, d), "q")
    _need(k, torch.bfloat16, (T, Hk, d), "k")
    _need(v, torch.bfloat16, (T, Hk, d), "v")
    _need(o, torch.bfloat16, (T, H, d), "o")
    _need(lse, torch.float32, (vl.sizes["lse"],), "lse")
    if tile_stats is not None:
        _need(tile_stats, torch.float32, (vl.sizes["tile_stats"],), "tile_stats")
    code = load().bl_attn_fwd_varlen(ctypes.byref(vl.struct), _ptr(q), _ptr(k), _ptr(v),
                                     float(scale), _ptr(o), _ptr(lse), _ptr(tile_stats),
                                     _stream(q.device))
    _check("bl_attn_fwd_varlen", code)


def mask_from_stats_varlen(vl: Varlen, tile_stats, lse, negl_prob, lists):
    z = vl.sizes
    _need(tile_stats, torch.float32, (z["tile_stats"],), "tile_stats")
    _need(lse, torch.float32, (z["lse"],), "lse")
    _need(lists["mask"], torch.uint8, (z["mask"],), "mask")
    _need(lists["kv_idx"], torch.int32, (z["mask"],), "kv_idx")
    _need(lists["kv_cnt"], torch.int32, (z["kv_cnt"],), "kv_cnt")
    _need(lists["q_idx"], torch.int32, (z["q_idx"],), "q_idx")
    _need(lists["q_cnt"], torch.int32, (z["q_cnt"],), "q_cnt")
    ls = _lists_struct(lists)
    code = load().bl_mask_from_stats_varlen(ctypes.byref(vl.struct), _ptr(tile_stats),
                                            _ptr(lse), float(negl_prob), ctypes.byref(ls),
                                            _stream(lse.device))
    _check("bl_mask_from_stats_varlen", code)


def fwd_tile_weights_supported_varlen(vl: Varlen) -> bool:
    """Whether bl_attn_fwd_tile_weights_varlen takes this batch (tiles of 64
    or 128, head dim 64 or 128, at most 2048 key tiles per sequence)."""
    longest = max(b - a for a, b in zip(vl.cu_seqlens[:-1], vl.cu_seqlens[1:]))
    return (vl.block_q in (64, 128) and vl.block_k in (64, 128) and vl.d in (64, 128)
            and -(-longest // vl.block_k) <= 2048)


def fwd_workspace_bytes_varlen(vl: Varlen) -> int:
    """Scratch of attn_fwd_tile_weights_varlen without a statistics output."""
    return int(load().bl_fwd_workspace_bytes_varlen(ctypes.byref(vl.struct)))


def attn_fwd_tile_weights_varlen(vl: Varlen, q, k, v, scale, o, lse, tile_logw, tile_stats=None,
                                 workspace=None):
    """bl_attn_fwd_tile_weights_varlen: tile_logw holds sizes["mask"] floats,
    laid out like the mask."""
    T, H, Hk, d = vl.total, vl.H, vl.Hk, vl.d
    _need(q, torch.bfloat16, (T, H, d), "q")
    _need(k, torch.bfloat16, (T, Hk, d), "k")
    _need(v, torch.bfloat16, (T, Hk, d), "v")
    _need(o, torch.bfloat16, (T, H, d), "o")
    _need(lse, torch.float32, (vl.sizes["lse"],), "lse")
    _need(tile_logw, torch.float32, (vl.sizes["mask"],), "tile_logw")
    if tile_stats is not None:
        _need(tile_stats, torch.float32, (vl.sizes["tile_stats"],), "tile_stats")
    nbytes = 0
    if workspace is not None:
        if workspace.dtype != torch.uint8 or not workspace.is_cuda:
            raise TypeError("workspace must be a CUDA uint8 tensor")
        nbytes = workspace.numel()
    code = load().bl_attn_fwd_tile_weights_varlen(
        ctypes.byref(vl.struct), _ptr(q), _ptr(k), _ptr(v), float(scale), _ptr(o), _ptr(lse),
        _ptr(tile_stats), _ptr(tile_logw), _ptr(workspace), nbytes, _stream(q.device))
    _check("bl_attn_fwd_tile_weights_varlen", code)


def mask_from_tile_weights_varlen(vl: Varlen, tile_logw, negl_prob, lists):
    z = vl.sizes
    _need(tile_logw, torch.float32, (z["mask"],), "tile_logw")
    _need(lists["mask"], torch.uint8, (z["mask"],), "mask")
    _need(lists["kv_idx"], torch.int32, (z["mask"],), "kv_idx")
    _need(lists["kv_cnt"], torch.int32, (z["kv_cnt"],), "kv_cnt")
    _need(lists["q_idx"], torch.int32, (z["q_idx"],), "q_idx")
    _need(lists["q_cnt"], torch.int32, (z["q_cnt"],), "q_cnt")
    ls = _lists_struct(lists)
    code = load().bl_mask_from_tile_weights_varlen(ctypes.byref(vl.struct), _ptr(tile_logw),
                                                   float(negl_prob), ctypes.byref(ls),
                                                   _stream(tile_logw.device))
    _check("bl_mask_from_tile_weights_varlen", code)


def attn_bwd_varlen(vl: Varlen, q, k, v, o, g_o, lse, scale, lists, g_q, g_k, g_v, workspace):
    T, H, Hk, d = vl.total, vl.H, vl.Hk, vl.d
    for t, nm, sh in ((q, "q", (T, H, d)), (k, "k", (T, Hk, d)), (v, "v", (T, Hk, d)),
                      (o, "o", (T, H, d)), (g_o, "g_o", (T, H, d)), (g_q, "g_q", (T, H, d)),
                      (g_k, "g_k", (T, Hk, d)), (g_v, "g_v", (T, Hk, d))):
        _need(t, torch.bfloat16, sh, nm)
    _need(lse, torch.float32, (vl.sizes["lse"],), "lse")
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA uint8 tensor")
    ls = None
    if lists is not None:
        _need(lists["q_idx"], torch.int32, (vl.sizes["q_idx"],), "q_idx")
        _need(lists["q_cnt"], torch.int32, (vl.sizes["q_cnt"],), "q_cnt")
        ls = _lists_struct(lists)
    code = load().bl_attn_bwd_varlen(ctypes.byref(vl.struct), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(o), _ptr(g_o), _ptr(lse), float(scale),
                                     ctypes.byref(ls) if ls is not None else None,
                                     _ptr(g_q), _ptr(g_k), _ptr(g_v), _ptr(workspace),
                                     workspace.numel(), _stream(q.device))
    _check("bl_attn_bwd_varlen", code)


def varlen_bwd_check_status(vl: Varlen, workspace) -> int:
    return int(load().bl_varlen_bwd_check_status(ctypes.byref(vl.struct), _ptr(workspace),
                                                 _stream(workspace.device)))
