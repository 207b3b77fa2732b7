"""The forward and the decode step inside a captured CUDA graph: after one
call outside the capture (which builds and uploads the cached plan and
reserves the library's workspaces), a call makes no synchronising or
allocating CUDA call, so it can be captured on the caller's stream; the
replayed graph reads the current contents of the captured buffers and
must give the eager result on new inputs."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from workloads import MaskSpec, bernoulli_causal_blocks, make_qkv  # noqa: E402

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


def _refill(ts, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    for t in ts:
        t.copy_(torch.randn(t.shape, generator=g, device="cuda").to(t.dtype))


@pytest.mark.parametrize("kind", ["sliding", "block", "column_major_copy"])
def test_forward_replays_in_a_graph(kind):
    B, H, N, d = 1, 4, 1024, 128
    q, k, v = make_qkv(B, H, N, d, "bf16", 1.0, 11, device="cuda")
    if kind == "sliding":
        spec = MaskSpec("sliding", [100, 37, 256, 8], sink=np.array([0.5, -1.0, 0.0, 2.0]))
    elif kind == "block":
        spec = MaskSpec("block", [128] * H, block=bernoulli_causal_blocks(H, N // 128, 3))
    else:  # an explicit order: the call runs the reorder pre-pass, then the kernel
        rng = np.random.default_rng(4)
        spec = MaskSpec("chunk", [128] * H, perm=[rng.permutation(N), None, None, None])
    mask = mattn.prepare(spec, H, N)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        mattn.attention(q, k, v, mask, out=out, lse=lse)  # plan, workspaces
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mattn.attention(q, k, v, mask, out=out, lse=lse)
    for seed in (21, 22):
        _refill((q, k, v), seed)
        graph.replay()
        ref_o, ref_l = mattn.attention(q, k, v, mask)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o), kind
        assert torch.equal(lse, ref_l), kind
    rc, word = mattn.device_status()
    assert rc == 0, f"device error word {word:#x}"


def test_decode_replays_in_a_graph():
    B, H, Hkv, L, d = 2, 8, 2, 3000, 128
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn((B, H, d), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((B, Hkv, L, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, Hkv, L, d), generator=g, device="cuda").to(torch.bfloat16)
    lens = torch.tensor([L, 1234], dtype=torch.int32, device="cuda")
    mask = mattn.prepare(MaskSpec("causal_window", [512] * H, sink_tokens=4), H, L)
    out = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        mattn.decode(q, k, v, mask, seq_lens=lens, out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mattn.decode(q, k, v, mask, seq_lens=lens, out=out, lse=lse)
    for seed, new_len in ((31, 2999), (32, 17)):
        _refill((q, k, v), seed)
        lens[1] = new_len  # the graph reads the lengths from device memory
        graph.replay()
        ref_o, ref_l = mattn.decode(q, k, v, mask, seq_lens=lens)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o)
        assert torch.equal(lse, ref_l)
