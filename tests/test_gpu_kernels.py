"""GPU checks of kernel building blocks: the FMA-pipe exp2 against CUDA's
exp2f, and the bounded-wait failure path (a wait that runs out returns an
error status instead of hanging, and the context stays usable)."""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import dense  # noqa: E402
from workloads import MaskSpec, make_qkv  # noqa: E402

pytestmark = pytest.mark.gpu
mattn = pytest.importorskip("block_sparse_attention_masked_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os

    if not os.path.exists(mattn.LIB_PATH):
        from block_sparse_attention_masked_gb300 import build

        build.build()
    mattn.lib()


def test_bounded_wait_reports_timeout_and_context_survives():
    L = mattn.lib()
    f = L.mattn_internal_fwd_wait_selftest
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.POINTER(mattn.MaskDesc), ctypes.c_void_p]
    n, d = 256, 64
    q, k, v = make_qkv(1, 1, n, d, "bf16", 1.0, seed=3, device="cuda")
    spec = MaskSpec("sliding", [32])
    mask = mattn.prepare(spec, 1, n)
    o = torch.zeros_like(q)
    lse = torch.zeros((1, 1, n), dtype=torch.float32, device="cuda")
    rc0, _ = mattn.device_status()
    assert rc0 == 0
    mattn.set_wait_timeout_ns(50_000_000)  # 50 ms
    try:
        stream = torch.cuda.current_stream().cuda_stream
        rc = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, n, d, mattn.BF16,
               ctypes.byref(mask.desc), stream)
        assert rc == 0
        rc, word = mattn.device_status()
        assert rc == mattn.ERR_TIMEOUT
        assert word & 0x10, hex(word)  # the self-test wait gave up
    finally:
        mattn.set_wait_timeout_ns(0)
    # the context is intact: a normal call still matches the oracle
    o2, lse2 = mattn.attention(q, k, v, mask)
    torch.cuda.synchronize()
    rc, word = mattn.device_status()
    assert rc == 0, hex(word)
    ref_o, _ = dense.attention(q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy(), spec)
    assert np.abs(o2.float().cpu().numpy()[0] - ref_o).max() < 2e-2
