"""Masked attention forward for GB300 (sm_103a): Python binding of libmattn.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libmattn.so`` behind the C ABI of ``include/mattn.h``.  PyTorch
provides device memory and streams.  There is no fallback: if the library
is missing or the device is not sm_103, the calls raise.

    import block_sparse_attention_masked_gb300 as mattn
    mask = mattn.prepare(spec, H=16, N=16384, device="cuda")
    o, lse = mattn.attention(q, k, v, mask)

``spec`` is a mask description with the attributes kind ("full", "chunk",
"sliding", "causal_window", "block"), head_param (per head C / w / W / Bs),
perm (per head None or an int array, perm[p] = token at position p),
perm_grid (per head None or (rows, cols) for the column-major walk of a
raster grid), block (bool [H, Nb, Nb]), sink (float [H] or None) and
sink_tokens (causal_window: the first sink_tokens positions stay visible).
k and v may have fewer heads than q (grouped-query attention).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmattn.so")
# The same library with device bounds checks compiled in (MATTN_DEBUG=1):
# loaded instead of LIB_PATH when the environment sets MATTN_DEBUG=1, or
# after use_debug_library(True).
DEBUG_LIB_PATH = os.path.join(_PKG, "libmattn_debug.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_CUDA = -3
ERR_TIMEOUT = -4
ERR_NO_DEVICE = -5
ERR_CAPACITY = -6
ERR_BOUNDS = -7
# device error-word bits of a failed debug check (mattn.h, "Debug library")
ERRW_BOUNDS = 1 << 5
ERRW_SITE = {"item": 1 << 8, "key_tile": 1 << 9, "load": 1 << 10, "store": 1 << 11, "order": 1 << 12,
             "ring": 1 << 13}

KIND = {"full": 0, "chunk": 1, "sliding": 2, "causal_window": 3, "block": 4}
BF16, F32 = 0, 1
ORDER_RASTER = -1
ORDER_COLUMN_MAJOR = -2
ORDER_BLOCK2X2_ROW = -3
ORDER_BLOCK2X2_COL = -4
_GRID_ORDERS = {"column_major": ORDER_COLUMN_MAJOR, "block2x2_row": ORDER_BLOCK2X2_ROW,
                "block2x2_col": ORDER_BLOCK2X2_COL}
TILE = 128
TILE_FULL, TILE_PARTIAL = 1, 2
FLAG_SCHEDULE_PAIRED, FLAG_SCHEDULE_SPLIT, FLAG_SCHEDULE_SINGLE, FLAG_SCHEDULE_PERSISTENT = 1, 2, 4, 8
RR_SINK_RECENT = 1
SCHEDULE = {None: 0, "auto": 0, "paired": FLAG_SCHEDULE_PAIRED, "split": FLAG_SCHEDULE_SPLIT,
            "single": FLAG_SCHEDULE_SINGLE, "persistent": FLAG_SCHEDULE_PERSISTENT}


class MattnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} ({code})")
        self.code = code


class MaskDesc(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("param", ctypes.c_int32),
        ("head_param", ctypes.POINTER(ctypes.c_int32)),
        ("head_order", ctypes.POINTER(ctypes.c_int32)),
        ("grid_rows", ctypes.c_int32),
        ("grid_cols", ctypes.c_int32),
        ("perm", ctypes.c_void_p),
        ("n_perm", ctypes.c_int32),
        ("block_bits", ctypes.c_void_p),
        ("block_heads", ctypes.c_int32),
        ("sink", ctypes.c_void_p),
        ("softmax_scale", ctypes.c_float),
        ("flags", ctypes.c_uint32),
        ("sink_tokens", ctypes.c_int32),
    ]


EXPORTS = (
    "mattn_fwd", "mattn_fwd_gqa", "mattn_fwd_host", "mattn_fwd_noalloc", "mattn_decode", "mattn_rr_select",
    "mattn_received",
    "mattn_count_pairs", "mattn_plan_schedule", "mattn_plan_tiles", "mattn_plan_tiles_device",
    "mattn_device_status", "mattn_debug_checks", "mattn_set_wait_timeout_ns", "mattn_status_string",
    "mattn_last_error", "mattn_version",
)

_lib = None
_libs = {}
_use_debug = os.environ.get("MATTN_DEBUG", "0") not in ("", "0")


def use_debug_library(on: bool = True) -> None:
    """Route every later call to libmattn_debug.so (on) or libmattn.so.
    Each library keeps its own device state (plans, workspaces, error
    word); both may be loaded in one process."""
    global _lib, _use_debug
    _use_debug = bool(on)
    _lib = None


def lib() -> ctypes.CDLL:
    """Load libmattn.so, or libmattn_debug.so (built by ``build.py`` /
    ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = DEBUG_LIB_PATH if _use_debug else LIB_PATH
    if path in _libs:
        _lib = _libs[path]
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} is not built ({path}); run "
                           "python -m block_sparse_attention_masked_gb300.build")
    L = ctypes.CDLL(path)
    vp, i32, u64p = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)
    dp = ctypes.POINTER(MaskDesc)
    L.mattn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, dp, vp]
    L.mattn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, dp, vp]
    L.mattn_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, dp, vp]
    L.mattn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, dp, vp]
    L.mattn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, dp, vp,
                                    ctypes.POINTER(ctypes.c_uint32)]
    L.mattn_rr_select.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, ctypes.c_float, ctypes.c_uint32,
                                  vp, vp, vp]
    L.mattn_received.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, dp, vp]
    L.mattn_count_pairs.argtypes = [dp, i32, i32, i32, u64p]
    L.mattn_plan_schedule.argtypes = [dp, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_uint32)]
    L.mattn_plan_tiles.argtypes = [dp, i32, i32, vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]
    L.mattn_plan_tiles_device.argtypes = [dp, i32, i32, vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t), vp]
    L.mattn_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.mattn_debug_checks.argtypes = []
    L.mattn_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    L.mattn_status_string.restype = ctypes.c_char_p
    L.mattn_status_string.argtypes = [i32]
    L.mattn_last_error.restype = ctypes.c_char_p
    L.mattn_last_error.argtypes = []
    L.mattn_version.argtypes = []
    for name in ("mattn_fwd", "mattn_fwd_gqa", "mattn_fwd_host", "mattn_fwd_noalloc", "mattn_decode", "mattn_rr_select", "mattn_received",
                 "mattn_count_pairs", "mattn_plan_schedule", "mattn_plan_tiles",
                 "mattn_plan_tiles_device", "mattn_device_status", "mattn_debug_checks",
                 "mattn_set_wait_timeout_ns", "mattn_version"):
        getattr(L, name).restype = ctypes.c_int
    _libs[path] = L
    _lib = L
    return L


def _check(rc: int) -> None:
    if rc != OK:
        L = lib()
        raise MattnError(rc, f"{L.mattn_status_string(rc).decode()}: {L.mattn_last_error().decode()}")


def pack_block_bits(block: np.ndarray) -> np.ndarray:
    """bool [Hb, Nb, Nb] -> uint64 [Hb, Nb, ceil(Nb/64)], bit n of row m = B[m][n]."""
    block = np.asarray(block, dtype=bool)
    if block.ndim == 2:
        block = block[None]
    hb, nb, nb2 = block.shape
    if nb != nb2:
        raise ValueError("block matrix must be square")
    wpr = (nb + 63) // 64
    padded = np.zeros((hb, nb, wpr * 64), dtype=bool)
    padded[:, :, :nb] = block
    by = np.packbits(padded.reshape(hb, nb, wpr, 64), axis=-1, bitorder="little")  # [hb, nb, wpr, 8]
    return by.view("<u8").reshape(hb, nb, wpr).copy()


class PreparedMask:
    """A mask descriptor plus the buffers it points at (kept alive here)."""

    def __init__(self, spec, H: int, N: int, device="cuda", scale: Optional[float] = None,
                 host_side: bool = False, schedule: Optional[str] = None):
        import torch

        self.H, self.N = H, N
        self.kind = spec.kind
        self._keep = []
        d = MaskDesc()
        d.kind = KIND[spec.kind]
        params = [int(x) for x in spec.head_param]
        if len(params) != H:
            raise ValueError("head_param must have H entries")
        d.param = params[0] if spec.kind != "full" else 0
        self._params = (ctypes.c_int32 * H)(*params)
        d.head_param = self._params
        orders = [ORDER_RASTER] * H
        grid = None
        explicit = []
        perms = getattr(spec, "perm", None)
        grids = getattr(spec, "perm_grid", None)
        for h in range(H):
            g = grids[h] if grids is not None else None
            pm = perms[h] if perms is not None else None
            if g is not None:
                gg = (int(g[0]), int(g[1]))
                if grid is not None and gg != grid:
                    raise ValueError("all grid-ordered heads must share one grid")
                grid = gg
                orders[h] = _GRID_ORDERS[g[2] if len(g) > 2 else "column_major"]
            elif pm is not None:
                orders[h] = len(explicit)
                explicit.append(np.asarray(pm, dtype=np.int32))
        self._orders = (ctypes.c_int32 * H)(*orders)
        d.head_order = self._orders
        if grid is not None:
            d.grid_rows, d.grid_cols = grid
        if explicit:
            arr = np.stack(explicit).astype(np.int32)
            t = torch.from_numpy(arr)
            t = t if host_side else t.to(device)
            self._keep.append(t)
            d.perm = t.data_ptr()
            d.n_perm = len(explicit)
        if spec.kind == "block":
            words = pack_block_bits(spec.block)
            self.block_words_host = words
            t = torch.from_numpy(words.view(np.int64))
            t = t if host_side else t.to(device)
            self._keep.append(t)
            d.block_bits = t.data_ptr()
            d.block_heads = words.shape[0]
        sink = getattr(spec, "sink", None)
        if sink is not None:
            t = torch.tensor(np.asarray(sink, dtype=np.float32))
            t = t if host_side else t.to(device)
            self._keep.append(t)
            d.sink = t.data_ptr()
        d.softmax_scale = 0.0 if scale is None else float(scale)
        if schedule not in SCHEDULE:
            raise ValueError(f"schedule must be one of {sorted(k for k in SCHEDULE if k)} or None")
        d.flags = SCHEDULE[schedule]
        d.sink_tokens = int(getattr(spec, "sink_tokens", 0) or 0)
        self.desc = d

    def host_desc(self):
        """A copy of the descriptor whose block bits point at host memory."""
        d = MaskDesc.from_buffer_copy(self.desc)
        if self.kind == "block":
            d.block_bits = self.block_words_host.ctypes.data
        d._owner = self  # the arrays the copied pointers refer to live in self
        return d


_SCHEDULE_NAMES = {FLAG_SCHEDULE_PAIRED: "paired", FLAG_SCHEDULE_SPLIT: "split", FLAG_SCHEDULE_SINGLE: "single",
                   FLAG_SCHEDULE_PERSISTENT: "persistent"}


def plan_schedule(mask: "PreparedMask", B: int, N: int, d: int, dtype: int = None) -> str:
    """The schedule the library runs for this mask and shape ("paired",
    "split", "single" or "persistent"); host only."""
    out = ctypes.c_uint32(0)
    _check(lib().mattn_plan_schedule(ctypes.byref(mask.desc), B, mask.H, N, d, BF16 if dtype is None else dtype,
                                     ctypes.byref(out)))
    return _SCHEDULE_NAMES[out.value]


def prepare(spec, H: int, N: int, device="cuda", scale: Optional[float] = None,
            schedule: Optional[str] = None) -> PreparedMask:
    """schedule: None / "auto" (library's choice), "paired", "split", "single"
    or "persistent" (the MATTN_FLAG_SCHEDULE_* flags); the result is the same
    up to rounding."""
    return PreparedMask(spec, H, N, device=device, scale=scale, schedule=schedule)


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def attention(q, k, v, mask: PreparedMask, out=None, lse=None, want_lse: bool = True, stream=None):
    """O, LSE of the masked attention forward on CUDA tensors [B, H, N, d]."""
    import torch

    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors (use attention_host for host buffers)")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous [B, H, N, d]")
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if (k.shape != (B, H_kv, N, d) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype
            or H % H_kv):
        raise ValueError("q [B, H, N, d] and k, v [B, H_kv, N, d] (H a multiple of H_kv) of one dtype")
    if out is None:
        out = torch.empty_like(q)
    if want_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
            lse.data_ptr() if lse is not None else None)
    if H_kv == H:
        rc = lib().mattn_fwd(*args, B, H, N, d, _dtype_code(q), ctypes.byref(mask.desc), stream)
    else:
        rc = lib().mattn_fwd_gqa(*args, B, H, H_kv, N, d, _dtype_code(q), ctypes.byref(mask.desc), stream)
    _check(rc)
    return out, lse


def decode(q, k_cache, v_cache, mask: PreparedMask, seq_lens=None, out=None, lse=None, want_lse: bool = True,
           stream=None):
    """One query per sequence against its key/value cache (``mattn_decode``).

    q: CUDA bf16 [B, H, d]; k_cache, v_cache: [B, H_kv, L, d]; seq_lens:
    CUDA int32 [B] (cached tokens with the new one; None = L).  ``mask``
    is prepared for H heads (kind "full" or "causal_window"; its N is not
    used).  Returns (o [B, H, d], lse [B, H] fp32 or None)."""
    import torch

    for t in (q, k_cache, v_cache):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k_cache and v_cache must be contiguous CUDA tensors")
    B, H, d = q.shape
    _, H_kv, L, _ = k_cache.shape
    if k_cache.shape != (B, H_kv, L, d) or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must be [B, H_kv, L, d]")
    if seq_lens is not None and (seq_lens.dtype != torch.int32 or seq_lens.shape != (B,) or not seq_lens.is_cuda):
        raise ValueError("seq_lens must be a CUDA int32 tensor [B]")
    if out is None:
        out = torch.empty_like(q)
    if want_lse and lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib().mattn_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                            lse.data_ptr() if lse is not None else None,
                            seq_lens.data_ptr() if seq_lens is not None else None,
                            B, H, H_kv, L, d, _dtype_code(q), ctypes.byref(mask.desc), stream)
    _check(rc)
    return out, lse


def attention_noalloc(q, k, v, mask: PreparedMask, out, lse=None, stream=None, check_wait: bool = True):
    """The same forward through ``mattn_fwd_noalloc``, which allocates no
    device memory: the caller passes ``out`` (and ``lse``) preallocated; the
    kernel's work list lives in a fixed static array of the library (bf16
    inputs read in place only; see the header for the limits).  With
    ``check_wait`` the call synchronises the stream and raises if a device
    wait gave up.  Returns (out, lse)."""
    import torch

    if not (q.is_cuda and k.is_cuda and v.is_cuda and out.is_cuda):
        raise ValueError("q, k, v and out must be CUDA tensors")
    for t in (q, k, v, out):
        if not t.is_contiguous():
            raise ValueError("q, k, v and out must be contiguous [B, H, N, d]")
    B, H, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or out.shape != q.shape:
        raise ValueError("q, k, v and out must have the same shape")
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    word = ctypes.c_uint32(0)
    rc = lib().mattn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 lse.data_ptr() if lse is not None else None, B, H, N, d, _dtype_code(q),
                                 ctypes.byref(mask.desc), stream, ctypes.byref(word) if check_wait else None)
    _check(rc)
    return out, lse


def unpack_block_bits(words: np.ndarray, nb: int) -> np.ndarray:
    """uint64 [..., Nb, ceil(Nb/64)] -> bool [..., Nb, Nb] (inverse of pack_block_bits)."""
    words = np.ascontiguousarray(np.asarray(words).view("<u8"))
    by = words.view(np.uint8).reshape(words.shape[:-1] + (words.shape[-1] * 8,))
    bits = np.unpackbits(by, axis=-1, bitorder="little")
    return bits[..., :nb].astype(bool)


def rr_select(q, k, stride: int = 8, block: int = 128, tau: float = 0.95, sink_recent: bool = False,
              want_scores: bool = False, stream=None):
    """RRAttention's dynamic block selection on CUDA bf16 tensors [B, H, N, d].

    Returns (bits, scores): bits int64 [B*H, Nb, ceil(Nb/64)] on the device,
    the block_bits layout of the attention mask (one [H, Nb, ..] slab per
    batch entry); scores fp32 [B*H, Nb, Nb] or None."""
    import torch

    if not (q.is_cuda and k.is_cuda):
        raise ValueError("q and k must be CUDA tensors")
    for t in (q, k):
        if not t.is_contiguous():
            raise ValueError("q and k must be contiguous [B, H, N, d]")
    B, H, N, d = q.shape
    if k.shape != q.shape or k.dtype != q.dtype:
        raise ValueError("q and k must have the same shape and dtype")
    if stride <= 0 or block % stride or N % stride:
        raise ValueError("the stride must divide N and the block size")
    nb = -(-(N // stride) // (block // stride))
    wpr = (nb + 63) // 64
    bits = torch.empty((B * H, nb, wpr), dtype=torch.int64, device=q.device)
    scores = torch.empty((B * H, nb, nb), dtype=torch.float32, device=q.device) if want_scores else None
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib().mattn_rr_select(q.data_ptr(), k.data_ptr(), B, H, N, d, _dtype_code(q), stride, block, float(tau),
                               RR_SINK_RECENT if sink_recent else 0, bits.data_ptr(),
                               scores.data_ptr() if scores is not None else None, stream)
    _check(rc)
    return bits, scores


class DeviceBlockMask:
    """A block-sparse mask descriptor over block bits already on the device
    (e.g. from rr_select): ``bits`` int64 [H, Nb, ceil(Nb/64)] for one batch
    entry, block size ``block``; optional per-head ``sink`` (fp32 [H] on the device)."""

    def __init__(self, bits, H: int, N: int, block: int, sink=None, schedule: Optional[str] = None):
        d = MaskDesc()
        d.kind = KIND["block"]
        d.param = int(block)
        self._params = (ctypes.c_int32 * H)(*([int(block)] * H))
        d.head_param = self._params
        d.block_bits = bits.data_ptr()
        d.block_heads = int(bits.shape[0])
        if sink is not None:
            d.sink = sink.data_ptr()
        d.softmax_scale = 0.0
        d.flags = SCHEDULE[schedule]
        self._keep = (bits, sink)
        self.desc = d
        self.H, self.N, self.kind = H, N, "block"


def received(q, k, lse, mask, out=None, stream=None):
    """Received attention r [B, H, N] (fp32, caller token order): the column
    sums of the attention matrix of the forward that wrote ``lse`` with the
    same q, k and mask."""
    import torch

    if not (q.is_cuda and k.is_cuda and lse.is_cuda):
        raise ValueError("q, k and lse must be CUDA tensors")
    for t in (q, k, lse):
        if not t.is_contiguous():
            raise ValueError("q, k and lse must be contiguous")
    B, H, N, d = q.shape
    if k.shape != q.shape or k.dtype != q.dtype or tuple(lse.shape) != (B, H, N) or lse.dtype != torch.float32:
        raise ValueError("k must match q; lse must be fp32 [B, H, N]")
    if out is None:
        out = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    _check(lib().mattn_received(q.data_ptr(), k.data_ptr(), lse.data_ptr(), out.data_ptr(), B, H, N, d,
                                _dtype_code(q), ctypes.byref(mask.desc), stream))
    return out


def attention_host(q, k, v, spec_or_mask, out=None, lse=None, stream=None):
    """The same on host (CPU, ideally pinned) tensors: copies in, computes, copies out."""
    import torch

    B, H, N, d = q.shape
    mask = spec_or_mask if isinstance(spec_or_mask, PreparedMask) else PreparedMask(
        spec_or_mask, H, N, host_side=True)
    desc = mask.host_desc()
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    rc = lib().mattn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                              B, H, N, d, _dtype_code(q), ctypes.byref(desc), stream)
    _check(rc)
    return out, lse


def count_pairs(spec_or_mask, B: int, H: int, N: int) -> int:
    mask = spec_or_mask if isinstance(spec_or_mask, PreparedMask) else PreparedMask(
        spec_or_mask, H, N, host_side=True)
    desc = mask.host_desc()
    out = ctypes.c_uint64(0)
    _check(lib().mattn_count_pairs(ctypes.byref(desc), B, H, N, ctypes.byref(out)))
    return int(out.value)


def plan_tiles(spec_or_mask, H: int, N: int) -> np.ndarray:
    """int32 [n, 4] (h, qt, kt, class) from the host planner."""
    mask = spec_or_mask if isinstance(spec_or_mask, PreparedMask) else PreparedMask(
        spec_or_mask, H, N, host_side=True)
    desc = mask.host_desc()
    n = ctypes.c_size_t(0)
    rc = lib().mattn_plan_tiles(ctypes.byref(desc), H, N, None, 0, ctypes.byref(n))
    if rc not in (OK, ERR_CAPACITY):
        _check(rc)
    buf = np.zeros((max(1, n.value), 4), dtype=np.int32)
    _check(lib().mattn_plan_tiles(ctypes.byref(desc), H, N, buf.ctypes.data, n.value, ctypes.byref(n)))
    return buf[:n.value]


def plan_tiles_device(mask: PreparedMask, H: int, N: int, stream=None) -> np.ndarray:
    """int32 [n, 4] from the device tile walker the attention kernel uses."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    n = ctypes.c_size_t(0)
    rc = lib().mattn_plan_tiles_device(ctypes.byref(mask.desc), H, N, None, 0, ctypes.byref(n), stream)
    if rc not in (OK, ERR_CAPACITY):
        _check(rc)
    buf = np.zeros((max(1, n.value), 4), dtype=np.int32)
    _check(lib().mattn_plan_tiles_device(ctypes.byref(mask.desc), H, N, buf.ctypes.data, n.value,
                                         ctypes.byref(n), stream))
    return buf[:n.value]


def device_status(stream=None):
    """(status, detail word); synchronises the stream and clears the device error word."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    word = ctypes.c_uint32(0)
    rc = lib().mattn_device_status(stream, ctypes.byref(word))
    return rc, int(word.value)


def set_wait_timeout_ns(ns: int) -> None:
    _check(lib().mattn_set_wait_timeout_ns(int(ns)))
