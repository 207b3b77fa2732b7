"""CPU checks of the debug library (libmattn_debug.so, the sources compiled
with MATTN_DEBUG=1) and of the host-side paths that keep a corrupted mask
description from reaching a kernel.

The debug library's device checks themselves run in test_gpu_debug.py; here:
it loads, exports what the header declares, says it is the debug build, and
its defect-planting test hook is refused by the product library.  Then the
host validation, in both libraries, of descriptors whose fields would index
out of range on the device (an explicit order past the orders passed, an
order code that does not exist, a grid that does not tile the sequence, a
bitmap head count that matches neither 1 nor H, no bitmap at all), and the
host planner's treatment of bitmap bits that must not matter (above the
diagonal, past the last block of a row).
"""

import ctypes
import os

import numpy as np
import pytest

from oracle import dense
from workloads import MaskSpec, bernoulli_causal_blocks

mattn = pytest.importorskip("block_sparse_attention_masked_gb300")

from test_abi_cpu import _declared_functions, _desc  # noqa: E402


@pytest.fixture(scope="module")
def libs():
    if not (os.path.exists(mattn.LIB_PATH) and os.path.exists(mattn.DEBUG_LIB_PATH)):
        from block_sparse_attention_masked_gb300 import build

        build.build()
    mattn.use_debug_library(True)
    dbg = mattn.lib()
    mattn.use_debug_library(False)
    prod = mattn.lib()
    yield {"product": prod, "debug": dbg}
    mattn.use_debug_library(False)


def test_debug_library_exports_and_identifies_itself(libs):
    names = _declared_functions()
    assert "mattn_debug_checks" in names
    for name in names:
        assert hasattr(libs["debug"], name), name
    assert libs["debug"].mattn_debug_checks() == 1
    assert libs["product"].mattn_debug_checks() == 0
    for L in libs.values():
        assert L.mattn_status_string(mattn.ERR_BOUNDS) == b"MATTN_ERR_BOUNDS"


def test_defect_hook_only_in_the_debug_library(libs):
    prod, dbg = libs["product"], libs["debug"]
    for L in (prod, dbg):
        L.mattn_internal_debug_corrupt.argtypes = [ctypes.c_int]
        L.mattn_internal_debug_corrupt.restype = ctypes.c_int
    assert prod.mattn_internal_debug_corrupt(1) == mattn.ERR_UNSUPPORTED
    assert dbg.mattn_internal_debug_corrupt(4) == mattn.ERR_INVALID_ARG
    assert dbg.mattn_internal_debug_corrupt(-1) == mattn.ERR_INVALID_ARG
    assert dbg.mattn_internal_debug_corrupt(2) == mattn.OK
    assert dbg.mattn_internal_debug_corrupt(0) == mattn.OK  # nothing left planted


def _rc(L, desc, H=2, N=256):
    out = ctypes.c_uint64(0)
    return L.mattn_count_pairs(ctypes.byref(desc), 1, H, N, ctypes.byref(out))


@pytest.mark.parametrize("which", ["product", "debug"])
def test_descriptors_that_would_index_out_of_range_are_refused(libs, which):
    """Each case names a field that the kernels use as an index; the host
    refuses it before anything is launched (MATTN_ERR_INVALID_ARG)."""
    L = libs[which]
    perm = ctypes.c_void_p(16)  # never read: validation fails first
    bits = np.zeros(8, np.uint64)
    cases = {
        "explicit order past n_perm": _desc(2, 3, head_order=(ctypes.c_int32 * 2)(1, -1), perm=perm, n_perm=1),
        "explicit order with n_perm 0": _desc(2, 3, head_order=(ctypes.c_int32 * 2)(0, -1), perm=perm, n_perm=0),
        "explicit order without perm": _desc(2, 3, head_order=(ctypes.c_int32 * 2)(0, -1), n_perm=1),
        "unknown order code": _desc(2, 3, head_order=(ctypes.c_int32 * 2)(-5, -1)),
        "column-major grid not tiling N": _desc(2, 3, head_order=(ctypes.c_int32 * 2)(-2, -1), grid_rows=16,
                                                grid_cols=8),
        "column-major grid negative": _desc(2, 3, head_order=(ctypes.c_int32 * 2)(-2, -1), grid_rows=-16,
                                            grid_cols=-16),
        "2x2 blocks on an odd grid": _desc(2, 3, head_order=(ctypes.c_int32 * 2)(-3, -1), grid_rows=1,
                                           grid_cols=256),
        "2x2 blocks grid not tiling N": _desc(2, 3, head_order=(ctypes.c_int32 * 2)(-4, -1), grid_rows=16,
                                              grid_cols=8),
        "head parameter 0": _desc(2, 3, head_param=(ctypes.c_int32 * 2)(3, 0)),
        "head parameter negative": _desc(1, 3, head_param=(ctypes.c_int32 * 2)(-7, 3)),
        "bitmap for 3 heads of 2": _desc(4, 128, block_bits=bits.ctypes.data, block_heads=3),
        "bitmap for 0 heads": _desc(4, 128, block_bits=bits.ctypes.data, block_heads=0),
        "block mask without a bitmap": _desc(4, 128, block_heads=1),
    }
    for name, desc in cases.items():
        assert _rc(L, desc) == mattn.ERR_INVALID_ARG, name
    # a block size that is no multiple of the 128-row tile: outside what is implemented
    assert _rc(L, _desc(4, 192, block_bits=bits.ctypes.data, block_heads=1)) == mattn.ERR_UNSUPPORTED
    assert _rc(L, _desc(2, 3), N=0) == mattn.ERR_INVALID_ARG
    assert _rc(L, _desc(2, 3), N=-5) == mattn.ERR_INVALID_ARG


@pytest.mark.parametrize("which", ["product", "debug"])
@pytest.mark.parametrize("n", [1000, 128 * 70])
def test_bitmap_bits_that_must_not_matter(libs, which, n):
    """Set bits above the diagonal (RRAttention Eq. 5: causality drops them)
    and in the padding past each row's last block change nothing in the
    host plan, which equals the oracle's enumeration of the clean bitmap."""
    L = libs[which]
    bs = 128
    nb = -(-n // bs)
    wpr = -(-nb // 64)
    clean = bernoulli_causal_blocks(1, nb, 7)
    spec = MaskSpec("block", [bs], block=clean)
    packed = mattn.pack_block_bits(clean)
    dirty = packed.copy()
    rng = np.random.default_rng(n)
    upper = np.triu(rng.random((nb, nb)) < 0.5, 1)
    dirty |= mattn.pack_block_bits(upper[None])
    if nb % 64:
        pad = ~np.uint64((1 << (nb % 64)) - 1)  # bits past column nb - 1 in the last word
        dirty[0, :, wpr - 1] |= pad
    assert (dirty != packed).any()

    def tiles(bits):
        desc = _desc(4, bs, block_bits=bits.ctypes.data, block_heads=1)
        cnt = ctypes.c_size_t(0)
        L.mattn_plan_tiles(ctypes.byref(desc), 1, n, None, 0, ctypes.byref(cnt))
        buf = np.zeros((max(1, cnt.value), 4), dtype=np.int32)
        assert L.mattn_plan_tiles(ctypes.byref(desc), 1, n, buf.ctypes.data, cnt.value, ctypes.byref(cnt)) == 0
        return [tuple(int(x) for x in t[1:]) for t in buf[:cnt.value]]

    want = dense.tile_list(spec, 0, n, 128)
    assert tiles(np.ascontiguousarray(packed)) == want
    assert tiles(np.ascontiguousarray(dirty)) == want
