"""mattn_fwd_noalloc, the forward for callers that must not allocate device
memory: a framework whose pooling allocator owns the device memory, a
serving loop that allows no cudaMalloc after start-up (it can synchronise
the device and take unbounded time), a plug-in host that gives the operator
no allocator.  That entry point keeps the kernel's work list, per-head
table and error word in a fixed static array of the library.  Here it is
called through the C ABI:

- compared with mattn_fwd on the same inputs, several calls in a row with
  different masks, so that whatever one call leaves in the shared array
  cannot leak into the next (each call synchronising, and again all queued
  on one stream without synchronising in between);
- compared with the fp64 oracle on sampled query rows, so that it stands on
  its own and not only on mattn_fwd;
- refused with MATTN_ERR_UNSUPPORTED on a stream under graph capture.

The file name sorts last so that a run stopping at the first failure has
run every other test before this one.
"""

import ctypes
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import dense  # noqa: E402
from workloads import (MaskSpec, bernoulli_causal_blocks, block2x2_order, column_major_order,  # noqa: E402
                       make_qkv)

mattn = pytest.importorskip("block_sparse_attention_masked_gb300")

MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3
MAX_HEADS = 4096
MAX_ITEMS = 65536


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(mattn.LIB_PATH):
        from block_sparse_attention_masked_gb300 import build

        build.build()
    return mattn.lib()


def _noalloc(q, k, v, mask, o, lse, word, stream=None):
    """One call through the C ABI; word None = asynchronous (no error-word read)."""
    B, H, N, d = q.shape
    s = (stream or torch.cuda.current_stream()).cuda_stream
    return mattn.lib().mattn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                         B, H, N, d, mattn.BF16, ctypes.byref(mask.desc), s,
                                         ctypes.byref(word) if word is not None else None)


def _compare(o, lse, o_ref, lse_ref, tag):
    a, b = o.float().cpu().numpy().astype(np.float64), o_ref.float().cpu().numpy().astype(np.float64)
    err = np.abs(a - b).max()
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    la, lb = lse.cpu().numpy().astype(np.float64), lse_ref.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isfinite(la), np.isfinite(lb)), f"{tag}: LSE -inf pattern differs"
    fin = np.isfinite(lb)
    lerr = np.abs(la[fin] - lb[fin]).max() if fin.any() else 0.0
    assert err <= MAX_ABS, f"{tag}: max abs {err:.3e}"
    assert rel <= REL_L2, f"{tag}: rel L2 {rel:.3e}"
    assert lerr <= LSE_ABS, f"{tag}: lse {lerr:.3e}"


def _cases():
    """Three launches of different shapes, masks, schedules and load modes,
    with the oracle's description of each (token orders as arrays)."""
    # A: block-sparse causal, split schedule, sink (16 work items)
    na, ha, da = 1024, 2, 128
    qa, ka, va = make_qkv(1, ha, na, da, "bf16", 1.0, seed=11, device="cuda")
    spec_a = MaskSpec("block", [128] * ha, block=bernoulli_causal_blocks(ha, na // 128, 11),
                      sink=np.array([0.75, -0.25]))
    # B: sliding window, heads 2-3 walked column-major over a 128 x 16 grid
    # (read through strided tensor maps), paired schedule (48 items)
    nb_, hb, db = 2048, 6, 80
    qb, kb, vb = make_qkv(1, hb, nb_, db, "bf16", 0.5, seed=12, device="cuda")
    grid = [None, None, (128, 16), (128, 16), None, None]
    spec_b = MaskSpec("sliding", [100, 37, 100, 256, 5, 1000], perm_grid=grid,
                      sink=np.linspace(-1.0, 1.0, hb))
    cm = column_major_order(128, 16)
    oracle_b = MaskSpec("sliding", spec_b.head_param, perm=[None, None, cm, cm, None, None], sink=spec_b.sink)
    # C: the two 2x2-block orders over a 64 x 64 grid, both read in place
    # through 5D tensor maps
    nc, hc, dc = 64 * 64, 2, 64
    qc, kc, vc = make_qkv(1, hc, nc, dc, "bf16", 1.0, seed=13, device="cuda")
    spec_c = MaskSpec("sliding", [90, 300],
                      perm=[block2x2_order(64, 64), block2x2_order(64, 64, by_columns=True)],
                      perm_grid=[(64, 64, "block2x2_row"), (64, 64, "block2x2_col")])
    return {"A": (qa, ka, va, mattn.prepare(spec_a, ha, na), spec_a),
            "B": (qb, kb, vb, mattn.prepare(spec_b, hb, nb_), oracle_b),
            "C": (qc, kc, vc, mattn.prepare(spec_c, hc, nc), spec_c)}


def _references(cases):
    refs = {name: mattn.attention(q, k, v, mask) for name, (q, k, v, mask, _) in cases.items()}
    torch.cuda.synchronize()
    assert mattn.device_status()[0] == 0
    return refs


def _empty_out(q):
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=q.device)
    return o, lse


@pytest.mark.gpu
def test_noalloc_matches_mattn_fwd_on_consecutive_calls(L):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    cases = _cases()
    refs = _references(cases)
    for i, name in enumerate(["A", "B", "C", "A", "B", "C"]):
        q, k, v, mask, _ = cases[name]
        o, lse = _empty_out(q)
        word = ctypes.c_uint32(0xFFFFFFFF)
        rc = _noalloc(q, k, v, mask, o, lse, word)
        assert rc == mattn.OK, f"call {i} ({name}): {L.mattn_status_string(rc)} {L.mattn_last_error()}"
        assert word.value == 0
        _compare(o, lse, *refs[name], tag=f"call {i} ({name})")


@pytest.mark.gpu
def test_noalloc_calls_queued_on_one_stream(L):
    """A, B, C, A queued on one stream without waiting for the error word:
    stream order alone keeps each call's work list apart from the next
    call's upload; every output must match mattn_fwd after one sync."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    cases = _cases()
    refs = _references(cases)
    order = ["A", "B", "C", "A"]
    outs = []
    for i, name in enumerate(order):
        q, k, v, mask, _ = cases[name]
        o, lse = _empty_out(q)
        rc = _noalloc(q, k, v, mask, o, lse, None)
        assert rc == mattn.OK, f"call {i} ({name}): {L.mattn_status_string(rc)} {L.mattn_last_error()}"
        outs.append((o, lse))
    torch.cuda.synchronize()
    for i, (name, (o, lse)) in enumerate(zip(order, outs)):
        _compare(o, lse, *refs[name], tag=f"queued call {i} ({name})")


@pytest.mark.gpu
def test_noalloc_matches_oracle_on_sampled_rows(L):
    """Each launch against the fp64 oracle on sampled query rows of every
    head: the first and last rows, rows at the 128-row tile edges, and
    random ones."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    rng = np.random.default_rng(7)
    for name, (q, k, v, mask, ospec) in _cases().items():
        o, lse = _empty_out(q)
        word = ctypes.c_uint32(0xFFFFFFFF)
        rc = _noalloc(q, k, v, mask, o, lse, word)
        assert rc == mattn.OK and word.value == 0, f"{name}: {L.mattn_last_error()}"
        n = q.shape[2]
        rows = np.unique(np.concatenate([[0, n - 1, 127, 128, n // 2 - 1, n // 2], rng.choice(n, 24, replace=False)]))
        ref_o, ref_lse = dense.attention(q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy(),
                                         ospec, rows=rows)
        H = q.shape[1]
        got_o = o.float().cpu().numpy().astype(np.float64)[0][:, rows].reshape(H, len(rows), -1)
        got_l = lse.cpu().numpy().astype(np.float64)[0][:, rows]
        err = np.abs(got_o - ref_o).max()
        rel = np.linalg.norm(got_o - ref_o) / np.linalg.norm(ref_o)
        assert err <= MAX_ABS, f"{name}: max abs {err:.3e}"
        assert rel <= REL_L2, f"{name}: rel L2 {rel:.3e}"
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(got_l), fin)
        assert np.abs(got_l[fin] - ref_lse[fin]).max() <= LSE_ABS, f"{name}: lse"


@pytest.mark.gpu
def test_noalloc_refuses_graph_capture(L):
    """On a stream under capture the call returns MATTN_ERR_UNSUPPORTED and
    records nothing; the capture then ends normally and its graph replays."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    q, k, v, mask, _ = _cases()["B"]
    o, lse = _empty_out(q)
    assert _noalloc(q, k, v, mask, o, lse, ctypes.c_uint32(0)) == mattn.OK  # eager first call
    side = torch.cuda.Stream()
    x = torch.zeros(64, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        x.add_(1.0)
        rc = _noalloc(q, k, v, mask, o, lse, None, stream=side)
    assert rc == mattn.ERR_UNSUPPORTED, L.mattn_status_string(rc)
    assert b"capture" in L.mattn_last_error()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.all(x == 1.0)


def _fake_ptr():
    # rejected calls return before any CUDA call: these are never dereferenced
    return ctypes.c_void_p(1 << 20)


def _call(L, desc, B, H, N, d, dtype=mattn.BF16):
    p = _fake_ptr()
    return L.mattn_fwd_noalloc(p, p, p, p, None, B, H, N, d, dtype, ctypes.byref(desc), None, None)


def test_noalloc_rejects_beyond_its_limits(L):
    full = mattn.MaskDesc()
    full.kind = mattn.KIND["full"]
    # B*H*ceil(ceil(N/128)/2) paired work items: 64*32*64 = 131072
    assert 64 * 32 * 64 > MAX_ITEMS
    assert _call(L, full, 64, 32, 16384, 128) == mattn.ERR_CAPACITY
    assert b"work items" in L.mattn_last_error()
    assert _call(L, full, 1, MAX_HEADS + 1, 128, 64) == mattn.ERR_CAPACITY
    assert b"heads" in L.mattn_last_error()
    # fp32 inputs and explicit token orders need a reorder buffer
    assert _call(L, full, 1, 2, 256, 64, dtype=mattn.F32) == mattn.ERR_UNSUPPORTED
    order = (ctypes.c_int32 * 2)(0, mattn.ORDER_RASTER)
    perm = (ctypes.c_int32 * 256)(*range(256))
    exp = mattn.MaskDesc()
    exp.kind = mattn.KIND["full"]
    exp.head_order = order
    exp.perm = ctypes.cast(perm, ctypes.c_void_p)
    exp.n_perm = 1
    assert _call(L, exp, 1, 2, 256, 64) == mattn.ERR_UNSUPPORTED
    # the usual argument checks still apply
    assert L.mattn_fwd_noalloc(None, None, None, None, None, 1, 2, 256, 64, mattn.BF16, ctypes.byref(full),
                               None, None) == mattn.ERR_INVALID_ARG
