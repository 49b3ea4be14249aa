"""Parity of the single-pass attention backward (attn_bwd_single_pass, d = 64:
one kernel per key block, dQ added into an fp32 buffer by bulk reduce-adds)
with the fp64 oracle, through the C ABI, and against the two-kernel path.

Tolerance: that of the two-kernel backward (test_bwd_gpu: max|err| <=
1e-2 max|ref|, mean|err| <= 4e-3 mean|ref| per tensor, against the fp64
gradients of the same bf16 inputs).  The single pass rounds P and dS to
bf16 exactly as the two-kernel path's dK/dV kernel does, so dK and dV must
equal that path's bit for bit; dQ sums the key blocks' fp32 shares in
arrival order, so it is held to the tolerance, not to bitwise equality.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_program_compilers_gb300 as pkg
from test_attn_gpu import rand
from test_bwd_gpu import REL_MAX, REL_MEAN, _check_grads, fp32_reference_grads

pytestmark = pytest.mark.gpu

D = 64


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg.build()
    torch.cuda.set_device(0)
    pkg.attn_get_status()


def run_both(q, k, v, g, causal, cu=None):
    """(single pass, two-kernel) gradients of the same inputs, as numpy."""
    dev = torch.device("cuda:0")
    tq, tk, tv, tg = (t.to(dev).contiguous() for t in (q, k, v, g))
    dcu = None if cu is None else torch.tensor(cu, device=dev)
    o, lse = pkg.attention(tq, tk, tv, causal=causal, cu_seqlens=dcu)
    if cu is None:
        B, N, Hq, d = q.shape
        Hkv = k.shape[2]
    else:
        N, Hq, d = q.shape
        Hkv = k.shape[1]
        B = len(cu) - 1
    out = []
    for single in (True, False):
        gq, gk, gv = (torch.full_like(t, float("nan")) for t in (tq, tk, tv))
        size = pkg.attn_bwd_single_pass_workspace_bytes if single else pkg.attn_bwd_workspace_bytes
        n = size(B, Hq, N, packed=cu is not None)
        ws = torch.full(((n + 15) // 16 * 4,), float("nan"), dtype=torch.float32, device=dev)
        run = pkg.attn_bwd_single_pass if single else pkg.attn_bwd
        run(tq, tk, tv, o, tg, lse, gq, gk, gv, B, Hq, Hkv, N, d, d ** -0.5, causal, dcu, ws)
        st = pkg.attn_get_status()
        assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
        out.append([t.float().cpu().numpy() for t in (gq, gk, gv)])
    return out


def check(q, k, v, g, causal, what, cu=None):
    if cu is None:
        B, N, Hq, d = q.shape
        Hkv = k.shape[2]
    else:
        N, Hq, d = q.shape
        Hkv = k.shape[1]
        B = len(cu) - 1
    single, two = run_both(q, k, v, g, causal, cu)
    refs = oracle.attn_bwd_oracle(q, k, v, g, B, Hq, Hkv, N, d, d ** -0.5, causal, cu_seqlens=cu)
    _check_grads(single, refs, what + " single pass")
    assert np.array_equal(single[1], two[1]), f"{what}: dk differs from the two-kernel path"
    assert np.array_equal(single[2], two[2]), f"{what}: dv differs from the two-kernel path"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 300, 513])
def test_single_pass_parity(causal, N):
    B, Hq, Hkv = 2, 4, 2
    q = rand((B, N, Hq, D), 101 + N)
    k = rand((B, N, Hkv, D), 102 + N)
    v = rand((B, N, Hkv, D), 103 + N)
    g = rand((B, N, Hq, D), 104 + N)
    check(q, k, v, g, causal, f"N={N} causal={causal}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (6, 3), (3, 3)])
def test_single_pass_gqa_groups(Hq, Hkv):
    B, N = 1, 384
    q, k, v = rand((B, N, Hq, D), 111), rand((B, N, Hkv, D), 112), rand((B, N, Hkv, D), 113)
    g = rand((B, N, Hq, D), 114)
    check(q, k, v, g, True, f"Hq={Hq} Hkv={Hkv}")


def test_single_pass_peaked_scores():
    B, N, H = 1, 640, 2
    q = rand((B, N, H, D), 121, 4.0)
    k, v, g = rand((B, N, H, D), 122), rand((B, N, H, D), 123), rand((B, N, H, D), 124)
    for causal in (False, True):
        check(q, k, v, g, causal, f"qx4 causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_single_pass_packed(causal):
    """Packed sequences of ragged lengths (an empty one, one-row ones, block
    edges): keys past a sequence's end must add nothing to any query's dQ."""
    lens = [1, 127, 128, 129, 300, 0, 513, 5]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, Hq, Hkv = int(cu[-1]), 4, 2
    q, k, v = rand((T, Hq, D), 131, 2.0), rand((T, Hkv, D), 132), rand((T, Hkv, D), 133)
    g = rand((T, Hq, D), 134)
    check(q, k, v, g, causal, f"packed causal={causal}", cu=cu)


def test_single_pass_long_sequences():
    """4096 rows (dK/dV units walking 32 query blocks of a four-head group,
    32 key blocks adding into every last query block's dQ), causal and not;
    the oracle's two calls run side by side."""
    from concurrent.futures import ThreadPoolExecutor
    Hq, Hkv, N = 4, 1, 4096
    cases = []
    for causal in (True, False):
        q, k, v = rand((1, N, Hq, D), 141 + causal), rand((1, N, Hkv, D), 142), rand((1, N, Hkv, D), 143)
        g = rand((1, N, Hq, D), 144)
        cases.append((q, k, v, g, causal))
    with ThreadPoolExecutor(len(cases)) as pool:
        futs = [pool.submit(oracle.attn_bwd_oracle, q, k, v, g, 1, Hq, Hkv, N, D, D ** -0.5, c)
                for q, k, v, g, c in cases]
        mines = [run_both(q, k, v, g, c) for q, k, v, g, c in cases]
        for (q, k, v, g, c), (single, two), fut in zip(cases, mines, futs):
            _check_grads(single, fut.result(), f"N={N} causal={c} single pass")
            assert np.array_equal(single[1], two[1]) and np.array_equal(single[2], two[2])


def test_single_pass_benchmarked_shape_fp32():
    """The benchmarked head-dim-64 backward (B2 Hq32 Hkv8 N4096 d64 causal)
    through the single pass, against the gradient formulas in fp32 on the
    GPU."""
    B, Hq, Hkv, N = 2, 32, 8, 4096
    gen = torch.Generator().manual_seed(2004)
    dev = torch.device("cuda:0")
    q, k, v, do = (torch.randn(s, generator=gen).to(torch.bfloat16).to(dev)
                   for s in ((B, N, Hq, D), (B, N, Hkv, D), (B, N, Hkv, D), (B, N, Hq, D)))
    o, lse = pkg.attention(q, k, v, causal=True)
    dq, dk, dv = pkg.attention_backward(q, k, v, o, lse, do, True, single_pass=True)
    assert pkg.attn_get_status() == pkg.ATTN_OK
    _check_grads([t.float().cpu().numpy() for t in (dq, dk, dv)],
                 fp32_reference_grads(q, k, v, do, True), "B2 Hq32 Hkv8 N4096 d64 causal")


def test_single_pass_repeat_close():
    """Two runs on the same inputs: dK, dV identical; dQ equal up to the
    order of the fp32 additions (far inside the tolerance)."""
    B, N, Hq, Hkv = 1, 1000, 4, 2
    q, k, v = rand((B, N, Hq, D), 151), rand((B, N, Hkv, D), 152), rand((B, N, Hkv, D), 153)
    g = rand((B, N, Hq, D), 154)
    a, _ = run_both(q, k, v, g, True)
    b, _ = run_both(q, k, v, g, True)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    scale = np.abs(a[0]).max()
    assert np.abs(a[0] - b[0]).max() <= 2 ** -7 * scale


def test_single_pass_rejects_other_head_dims_and_small_workspace():
    B, N, H = 1, 256, 2
    dev = torch.device("cuda:0")
    lse = torch.zeros((B, H, N), dtype=torch.float32, device=dev)
    for d in (128, 256):
        t = torch.zeros((B, N, H, d), dtype=torch.bfloat16, device=dev)
        n = pkg.attn_bwd_single_pass_workspace_bytes(B, H, N)
        ws = torch.empty(((n + 15) // 16 * 4,), dtype=torch.float32, device=dev)
        rc = pkg.attn_bwd_single_pass(t, t, t, t, t, lse, t, t, t, B, H, H, N, d, 0.125, True,
                                      workspace=ws, check=False)
        assert rc == pkg.ATTN_ERR_INVALID_ARG
    t = torch.zeros((B, N, H, D), dtype=torch.bfloat16, device=dev)
    n = pkg.attn_bwd_workspace_bytes(B, H, N)   # the two-kernel path's: too small here
    ws = torch.empty(((n + 15) // 16 * 4,), dtype=torch.float32, device=dev)
    rc = pkg.attn_bwd_single_pass(t, t, t, t, t, lse, t, t, t, B, H, H, N, D, 0.125, True,
                                  workspace=ws, check=False)
    assert rc == pkg.ATTN_ERR_INVALID_ARG


def test_single_pass_bad_offsets_reported():
    T, H = 300, 2
    dev = torch.device("cuda:0")
    t = rand((T, H, D), 161).to(dev)
    lse = torch.zeros((H, T), dtype=torch.float32, device=dev)
    out = torch.full_like(t, float("nan"))
    bad = torch.tensor([0, 200, 100], dtype=torch.int32, device=dev)   # decreasing
    n = pkg.attn_bwd_single_pass_workspace_bytes(2, H, T, packed=True)
    ws = torch.empty(((n + 15) // 16 * 4,), dtype=torch.float32, device=dev)
    pkg.attn_bwd_single_pass(t, t, t, t, t, lse, out, out, out, 2, H, H, T, D, 0.125, True, bad,
                             ws)
    assert pkg.attn_get_status() == pkg.ATTN_ERR_BAD_SEQLENS
    assert torch.isnan(out.float()).all()
