"""Parity of the attention backward (attn_bwd: dQ, dK, dV) with the fp64
oracle, through the C ABI.

Tolerance (derived, the task states none for gradients): the kernels round
P and dS to bf16 before the products (relative error <= 2^-9 per term) and
round dQ, dK, dV to bf16 at the end (relative half-ulp <= 2^-8); per tensor
max|err| <= 1e-2 * max|ref| and mean|err| <= 4e-3 * mean|ref| against the
fp64 gradients of the same bf16 inputs (observed about 0.3-0.45% and 0.25%),
with the scale floored at 1e-3 for gradients that are exactly zero.
Outputs are NaN-filled before every call and must come back finite.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_program_compilers_gb300 as pkg
from test_attn_gpu import rand

pytestmark = pytest.mark.gpu

REL_MAX, REL_MEAN = 1e-2, 4e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg.build()
    torch.cuda.set_device(0)
    pkg.attn_get_status()


def run_bwd(q, k, v, g, causal):
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    dev = torch.device("cuda:0")
    dq_, dk_, dv_, dg = (t.to(dev).contiguous() for t in (q, k, v, g))
    o, lse = pkg.attention(dq_, dk_, dv_, causal=causal)
    gq = torch.full_like(dq_, float("nan"))
    gk = torch.full_like(dk_, float("nan"))
    gv = torch.full_like(dv_, float("nan"))
    n = pkg.attn_bwd_workspace_bytes(B, Hq, N)
    ws = torch.full(((n + 15) // 16 * 4,), float("nan"), dtype=torch.float32, device=dev)
    pkg.attn_bwd(dq_, dk_, dv_, o, dg, lse, gq, gk, gv, B, Hq, Hkv, N, d, d ** -0.5, causal,
                 workspace=ws)
    st = pkg.attn_get_status()
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    return [t.float().cpu().numpy() for t in (gq, gk, gv)]


def check(q, k, v, g, causal, what):
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    mine = run_bwd(q, k, v, g, causal)
    refs = oracle.attn_bwd_oracle(q, k, v, g, B, Hq, Hkv, N, d, d ** -0.5, causal)
    for name, m, r in zip(("dq", "dk", "dv"), mine, refs):
        assert np.isfinite(m).all(), f"{what} {name}: unwritten or non-finite"
        err = np.abs(m - r)
        msg = (f"{what} {name}: max|err|={err.max():.3e} (max|ref| {np.abs(r).max():.3e}) "
               f"mean|err|={err.mean():.3e} (mean|ref| {np.abs(r).mean():.3e})")
        # (a gradient that is exactly zero, e.g. dQ with one visible key,
        # is held to 1e-3 of an absolute scale of one)
        assert err.max() <= REL_MAX * max(np.abs(r).max(), 1e-3), msg
        assert err.mean() <= REL_MEAN * max(np.abs(r).mean(), 1e-3), msg


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 300, 513])
def test_bwd_parity(d, causal, N):
    B, Hq, Hkv = 2, 4, 2
    q = rand((B, N, Hq, d), 1 + N + d)
    k = rand((B, N, Hkv, d), 2 + N + d)
    v = rand((B, N, Hkv, d), 3 + N + d)
    g = rand((B, N, Hq, d), 4 + N + d)
    check(q, k, v, g, causal, f"d={d} N={N} causal={causal}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (6, 3), (3, 3)])
def test_bwd_gqa_groups(Hq, Hkv):
    B, N, d = 1, 384, 128
    q, k, v = rand((B, N, Hq, d), 11), rand((B, N, Hkv, d), 12), rand((B, N, Hkv, d), 13)
    g = rand((B, N, Hq, d), 14)
    check(q, k, v, g, True, f"Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (3, 3)])
def test_bwd_gqa_groups_d256(Hq, Hkv):
    """Head dim 256 (three kernels: dV, dK, dQ) with grouped heads."""
    B, N, d = 1, 384, 256
    q, k, v = rand((B, N, Hq, d), 15), rand((B, N, Hkv, d), 16), rand((B, N, Hkv, d), 17)
    g = rand((B, N, Hq, d), 18)
    check(q, k, v, g, True, f"d=256 Hq={Hq} Hkv={Hkv}")


def test_bwd_peaked_scores():
    B, N, H, d = 1, 640, 2, 64
    q = rand((B, N, H, d), 21, 4.0)
    k, v, g = rand((B, N, H, d), 22), rand((B, N, H, d), 23), rand((B, N, H, d), 24)
    for causal in (False, True):
        check(q, k, v, g, causal, f"qx4 causal={causal}")


def test_bwd_deterministic():
    B, N, Hq, Hkv, d = 1, 700, 4, 2, 128
    q, k, v = rand((B, N, Hq, d), 31), rand((B, N, Hkv, d), 32), rand((B, N, Hkv, d), 33)
    g = rand((B, N, Hq, d), 34)
    a = run_bwd(q, k, v, g, True)
    b = run_bwd(q, k, v, g, True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_bwd_small_workspace_rejected():
    B, N, H, d = 1, 256, 2, 64
    dev = torch.device("cuda:0")
    t = torch.zeros((B, N, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((B, H, N), dtype=torch.float32, device=dev)
    ws = torch.empty((16,), dtype=torch.float32, device=dev)
    rc = pkg.attn_bwd(t, t, t, t, t, lse, t, t, t, B, H, H, N, d, 0.125, True, workspace=ws,
                      check=False)
    assert rc == pkg.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_packed(d, causal):
    lens = [1, 127, 128, 129, 300, 0, 513, 5]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, Hq, Hkv = int(cu[-1]), 4, 2
    q, k, v = rand((T, Hq, d), 41 + d, 2.0), rand((T, Hkv, d), 42 + d), rand((T, Hkv, d), 43 + d)
    g = rand((T, Hq, d), 44 + d)
    dev = torch.device("cuda:0")
    dcu = torch.tensor(cu, device=dev)
    dq_, dk_, dv_, dg = (t.to(dev) for t in (q, k, v, g))
    o, lse = pkg.attention(dq_, dk_, dv_, causal=causal, cu_seqlens=dcu)
    grads = pkg.attention_backward(dq_, dk_, dv_, o, lse, dg, causal, cu_seqlens=dcu)
    assert pkg.attn_get_status() == pkg.ATTN_OK
    refs = oracle.attn_bwd_oracle(q, k, v, g, len(lens), Hq, Hkv, T, d, d ** -0.5, causal,
                                  cu_seqlens=cu)
    for name, m, r in zip(("dq", "dk", "dv"), grads, refs):
        m = m.float().cpu().numpy()
        assert np.isfinite(m).all()
        err = np.abs(m - r)
        assert err.max() <= REL_MAX * max(np.abs(r).max(), 1e-3), (name, err.max())
        assert err.mean() <= REL_MEAN * max(np.abs(r).mean(), 1e-3), (name, err.mean())


def test_bwd_packed_bad_offsets_reported():
    T, H, d = 300, 2, 64
    dev = torch.device("cuda:0")
    t = rand((T, H, d), 51).to(dev)
    lse = torch.zeros((H, T), dtype=torch.float32, device=dev)
    out = torch.full_like(t, float("nan"))
    bad = torch.tensor([0, 200, 100], dtype=torch.int32, device=dev)   # decreasing
    n = pkg.attn_bwd_workspace_bytes(2, H, T, packed=True)
    ws = torch.empty(((n + 15) // 16 * 4,), dtype=torch.float32, device=dev)
    pkg.attn_bwd(t, t, t, t, t, lse, out, out, out, 2, H, H, T, d, 0.125, True, bad, ws)
    assert pkg.attn_get_status() == pkg.ATTN_ERR_BAD_SEQLENS
    assert torch.isnan(out.float()).all()


def _oracle_async(pool, q, k, v, g, B, Hq, Hkv, N, d, causal, cu=None):
    return pool.submit(oracle.attn_bwd_oracle, q, k, v, g, B, Hq, Hkv, N, d, d ** -0.5,
                       causal, cu_seqlens=cu)


def _check_grads(mine, refs, what):
    for name, m, r in zip(("dq", "dk", "dv"), mine, refs):
        assert np.isfinite(m).all(), f"{what} {name}: unwritten or non-finite"
        err = np.abs(m - r)
        msg = (f"{what} {name}: max|err|={err.max():.3e} (max|ref| {np.abs(r).max():.3e}) "
               f"mean|err|={err.mean():.3e} (mean|ref| {np.abs(r).mean():.3e})")
        assert err.max() <= REL_MAX * max(np.abs(r).max(), 1e-3), msg
        assert err.mean() <= REL_MEAN * max(np.abs(r).mean(), 1e-3), msg


def test_bwd_parity_long_sequences():
    """Sequences as long as the benchmarked backward's (4096 rows): dK/dV
    units that walk 32 query blocks of every query head of a four-head group,
    dQ units that walk 32 key blocks; causal at N = 4096, non-causal at
    N = 2048, and a packed batch whose first sequence is longer than 4096.
    One kv head keeps the fp64 oracle to seconds; its three calls run
    side by side (the C oracle releases the interpreter lock)."""
    from concurrent.futures import ThreadPoolExecutor
    d, Hq, Hkv = 128, 4, 1
    cases = []
    for N, causal in ((4096, True), (2048, False)):
        q, k, v = rand((1, N, Hq, d), 61 + N), rand((1, N, Hkv, d), 62 + N), rand((1, N, Hkv, d), 63 + N)
        g = rand((1, N, Hq, d), 64 + N)
        cases.append((f"N={N} causal={causal}", (q, k, v, g, 1, N, causal, None)))
    lens = [4500, 300, 1, 129]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, g = rand((T, Hq, d), 71, 2.0), rand((T, Hkv, d), 72), rand((T, Hkv, d), 73), rand((T, Hq, d), 74)
    cases.append(("packed, first sequence 4500", (q, k, v, g, len(lens), T, True, cu)))
    with ThreadPoolExecutor(len(cases)) as pool:
        futs = [_oracle_async(pool, q_, k_, v_, g_, B_, Hq, Hkv, N_, d, c_, cu_)
                for _, (q_, k_, v_, g_, B_, N_, c_, cu_) in cases]
        dev = torch.device("cuda:0")
        mines = []
        for what, (q_, k_, v_, g_, B_, N_, c_, cu_) in cases:
            if cu_ is None:
                mines.append(run_bwd(q_, k_, v_, g_, c_))
                continue
            dcu = torch.tensor(cu_, device=dev)
            tq, tk, tv, tg = (t.to(dev) for t in (q_, k_, v_, g_))
            o, lse = pkg.attention(tq, tk, tv, causal=c_, cu_seqlens=dcu)
            grads = pkg.attention_backward(tq, tk, tv, o, lse, tg, c_, cu_seqlens=dcu)
            assert pkg.attn_get_status() == pkg.ATTN_OK
            mines.append([t.float().cpu().numpy() for t in grads])
        for (what, _), mine, fut in zip(cases, mines, futs):
            _check_grads(mine, fut.result(), what)


def test_bwd_d256_long_sequences():
    """Head dim 256 at 2048 rows (16 query blocks per dK/dV unit and per dQ
    unit), causal and not, against the fp64 oracle."""
    from concurrent.futures import ThreadPoolExecutor
    d, Hq, Hkv, N = 256, 2, 1, 2048
    cases = []
    for causal in (True, False):
        q, k, v = rand((1, N, Hq, d), 81 + causal), rand((1, N, Hkv, d), 82), rand((1, N, Hkv, d), 83)
        g = rand((1, N, Hq, d), 84)
        cases.append((f"d=256 N={N} causal={causal}", (q, k, v, g, causal)))
    with ThreadPoolExecutor(len(cases)) as pool:
        futs = [_oracle_async(pool, q_, k_, v_, g_, 1, Hq, Hkv, N, d, c_, None)
                for _, (q_, k_, v_, g_, c_) in cases]
        mines = [run_bwd(q_, k_, v_, g_, c_) for _, (q_, k_, v_, g_, c_) in cases]
        for (what, _), mine, fut in zip(cases, mines, futs):
            _check_grads(mine, fut.result(), what)


def fp32_reference_grads(q, k, v, do, causal):
    """The gradient formulas in fp32 with PyTorch on the GPU, head by head
    (TF32 off): S = scale Q K^T (masked), P = softmax(S), dP = dO V^T,
    D = rowsum(P dP), dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q,
    dV = P^T dO, with dK and dV summed over each kv head's query heads."""
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    dev = q.device
    scale = d ** -0.5
    grp = Hq // Hkv
    mask = torch.ones(N, N, dtype=torch.bool, device=dev).triu(1) if causal else None
    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        rq = torch.empty((B, N, Hq, d), dtype=torch.float32, device=dev)
        rk = torch.zeros((B, N, Hkv, d), dtype=torch.float32, device=dev)
        rv = torch.zeros((B, N, Hkv, d), dtype=torch.float32, device=dev)
        for b in range(B):
            for h in range(Hq):
                kv = h // grp
                qh, kh, vh, gh = (q[b, :, h].float(), k[b, :, kv].float(), v[b, :, kv].float(),
                                  do[b, :, h].float())
                sc = qh @ kh.T * scale
                if mask is not None:
                    sc = sc.masked_fill(mask, float("-inf"))
                p = torch.softmax(sc, -1)
                del sc
                dp = gh @ vh.T
                ds = p * (dp - (p * dp).sum(-1, keepdim=True))
                rq[b, :, h] = scale * (ds @ kh)
                rk[b, :, kv] += scale * (ds.T @ qh)
                rv[b, :, kv] += p.T @ gh
                del p, dp, ds
    finally:
        torch.backends.cuda.matmul.allow_tf32 = tf32
    return [t.cpu().numpy() for t in (rq, rk, rv)]


def test_bwd_d256_long_shape_fp32():
    """The long head-dim-256 configuration's shape (B1 Hq16 Hkv2 N16384 d256
    causal, the shape of the benchmarked d = 256 backward) against the fp32
    gradient formulas on the GPU."""
    B, Hq, Hkv, N, d = 1, 16, 2, 16384, 256
    gen = torch.Generator().manual_seed(2005)
    dev = torch.device("cuda:0")
    q, k, v, do = (torch.randn(s, generator=gen).to(torch.bfloat16).to(dev)
                   for s in ((B, N, Hq, d), (B, N, Hkv, d), (B, N, Hkv, d), (B, N, Hq, d)))
    o, lse = pkg.attention(q, k, v, causal=True)
    dq, dk, dv = pkg.attention_backward(q, k, v, o, lse, do, True)
    assert pkg.attn_get_status() == pkg.ATTN_OK
    _check_grads([t.float().cpu().numpy() for t in (dq, dk, dv)],
                 fp32_reference_grads(q, k, v, do, True), "B1 Hq16 Hkv2 N16384 d256 causal")


def test_bwd_benchmarked_shape_fp32():
    """The benchmarked backward itself (B2 Hq32 Hkv8 N4096 d128 causal)
    against the gradient formulas in fp32 on the GPU (the reference's own
    error is far below the tolerance)."""
    B, Hq, Hkv, N, d = 2, 32, 8, 4096, 128
    gen = torch.Generator().manual_seed(2004)
    dev = torch.device("cuda:0")
    q, k, v, do = (torch.randn(s, generator=gen).to(torch.bfloat16).to(dev)
                   for s in ((B, N, Hq, d), (B, N, Hkv, d), (B, N, Hkv, d), (B, N, Hq, d)))
    o, lse = pkg.attention(q, k, v, causal=True)
    dq, dk, dv = pkg.attention_backward(q, k, v, o, lse, do, True)
    assert pkg.attn_get_status() == pkg.ATTN_OK
    _check_grads([t.float().cpu().numpy() for t in (dq, dk, dv)],
                 fp32_reference_grads(q, k, v, do, True), "B2 Hq32 Hkv8 N4096 d128 causal")
