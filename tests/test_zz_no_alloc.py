"""attn_fwd_decode_static (the allocation-free decode entry point, fixed
device scratch) against attn_fwd_decode with a caller workspace.

Collected last on purpose: it must pass on its own and after every other
test has used the library on this device.
"""
import numpy as np
import pytest
import torch

import tensor_program_compilers_gb300 as pkg

pytestmark = pytest.mark.gpu


def rand(shape, seed, mult=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * mult).to(torch.bfloat16)


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg.build()
    torch.cuda.set_device(0)
    pkg.attn_get_status()


def problem(B, Nq, Hq, Hkv, Nk, d, seed, lens):
    dev = torch.device("cuda:0")
    q = rand((B, Nq, Hq, d), seed, 2.0).to(dev)
    k = rand((B, Nk, Hkv, d), seed + 1).to(dev)
    v = rand((B, Nk, Hkv, d), seed + 2).to(dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    return q, k, v, sl


@pytest.mark.parametrize("d,causal,Nq", [(64, False, 1), (128, True, 4), (256, True, 2)])
def test_static_matches_workspace_entry_point_twice(d, causal, Nq):
    B, Hq, Hkv, Nk = 3, 16, 4, 4000
    lens = [4000, 1234, Nq]
    q, k, v, sl = problem(B, Nq, Hq, Hkv, Nk, d, 10 + d, lens)
    n = pkg.attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d)
    assert 0 < n <= pkg.DECODE_STATIC_SCRATCH_BYTES
    ws = torch.empty(((n + 15) // 16 * 4,), dtype=torch.float32, device="cuda:0")
    o_ref = torch.full_like(q, float("nan"))
    l_ref = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device="cuda:0")
    pkg.attn_fwd_decode(q, k, v, o_ref, l_ref, B, Hq, Hkv, Nq, Nk, d, d ** -0.5, causal, sl, ws)
    assert pkg.attn_get_status() == pkg.ATTN_OK
    for call in range(2):   # two calls in a row reuse the same scratch
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device="cuda:0")
        pkg.attn_fwd_decode_static(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, d ** -0.5, causal, sl)
        assert pkg.attn_get_status() == pkg.ATTN_OK
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)), f"call {call}: O differs"
        assert torch.equal(lse, l_ref), f"call {call}: LSE differs"


def test_static_rejects_problems_larger_than_its_scratch():
    """A problem whose partial states exceed the fixed scratch is refused
    before anything runs.  The split count follows the SM count (one
    sequence, one kv head, keys enough for a split per SM), so the problem is
    built from the device: its states take about SMs x 128 rows x 257 floats,
    past 8 MiB on any part with more than 64 SMs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, Nq, Hq, Hkv, d = 1, 8, 16, 1, 256
    Nk = 128 * max(sms, 1) * 2
    n = pkg.attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d)
    if n <= pkg.DECODE_STATIC_SCRATCH_BYTES:
        pytest.skip(f"{sms} SMs: no decode problem needs more than the fixed scratch")
    dev = torch.device("cuda:0")
    q = torch.zeros((B, Nq, Hq, d), dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    k = torch.zeros((1, 16, Hkv, d), dtype=torch.bfloat16, device=dev)   # never read
    rc = pkg.attn_fwd_decode_static(q, k, k, o, lse, B, Hq, Hkv, Nq, Nk, d, 0.1, False,
                                    check=False)
    assert rc == pkg.ATTN_ERR_INVALID_ARG


def test_static_single_split_needs_no_scratch():
    B, Nq, Hq, Hkv, Nk, d = 64, 1, 16, 8, 256, 64
    assert pkg.attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d) == 0
    lens = [256 - (b * 5) % 200 for b in range(B)]
    q, k, v, sl = problem(B, Nq, Hq, Hkv, Nk, d, 40, lens)
    o_ref, l_ref = pkg.decode(q, k, v, causal=False, seqlens_k=sl)
    o = torch.empty_like(q)
    lse = torch.empty_like(l_ref)
    pkg.attn_fwd_decode_static(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, d ** -0.5, False, sl)
    assert pkg.attn_get_status() == pkg.ATTN_OK
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse, l_ref)


@pytest.mark.parametrize("Nq,Hq", [(1, 16), (4, 16)])
def test_static_decode_replays_in_a_cuda_graph(Nq, Hq):
    """The entry point's purpose: after one call outside capture it needs no
    allocation and no host lookup, so it can be captured in a CUDA graph.
    Two replays give the workspace entry point's bits (group 4 x Nq 1: the
    CUDA-core kernel with key splits and the merge; Nq 4: the tile kernel)."""
    B, Hkv, Nk, d = 3, 4, 3000, 128
    lens = [3000, 1500, Nq]
    q, k, v, sl = problem(B, Nq, Hq, Hkv, Nk, d, 90 + Nq, lens)
    n = pkg.attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d)
    assert 0 < n <= pkg.DECODE_STATIC_SCRATCH_BYTES
    ws = torch.empty(((n + 15) // 16 * 4,), dtype=torch.float32, device="cuda:0")
    o_ref = torch.full_like(q, float("nan"))
    l_ref = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device="cuda:0")
    pkg.attn_fwd_decode(q, k, v, o_ref, l_ref, B, Hq, Hkv, Nq, Nk, d, d ** -0.5, True, sl, ws)
    assert pkg.attn_get_status() == pkg.ATTN_OK
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device="cuda:0")
    call = lambda: pkg.attn_fwd_decode_static(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, d ** -0.5,
                                              True, sl)
    call()   # the first call outside capture (device set-up)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            call()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pkg.attn_get_status() == pkg.ATTN_OK
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse, l_ref)
