"""Parity of the split-key decode path (attn_fwd_decode: partial states per
key split, merged by a second kernel) with the fp64 oracle in the decode
convention, through the C ABI.  Same tolerances as test_attn_gpu.py."""
import numpy as np
import pytest
import torch

import oracle
import tensor_program_compilers_gb300 as pkg
from test_attn_gpu import compare, rand

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg.build()
    torch.cuda.set_device(0)
    pkg.attn_get_status()


def caches(B, Nk, Hkv, d, lens, seed):
    """Key/value caches whose rows past each length hold finite decoys
    (large keys that would dominate if they were not masked)."""
    k = rand((B, Nk, Hkv, d), seed)
    v = rand((B, Nk, Hkv, d), seed + 1)
    for b, L in enumerate(lens):
        k[b, L:] = 8.0
        v[b, L:] = 100.0
    return k, v


def run_decode(q, k, v, lens, causal, scale, check_status=True):
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    dev = torch.device("cuda:0")
    dq, dk, dv = (t.to(dev).contiguous() for t in (q, k, v))
    sl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=dev)
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device=dev)
    n = pkg.attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d)
    ws = torch.full(((max(n, 16) + 15) // 16 * 4,), float("nan"), dtype=torch.float32, device=dev)
    rc = pkg.attn_fwd_decode(dq, dk, dv, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, sl, ws,
                             check=False)
    assert rc == pkg.ATTN_OK, pkg.attn_status_string(rc)
    st = pkg.attn_get_status()
    if check_status:
        assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    return o.float().cpu().numpy(), lse.cpu().numpy(), n


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq", [1, 4])
def test_decode_parity(d, causal, Nq):
    B, Hq, Hkv, Nk = 3, 8, 2, 3000
    lens = [3000, 1, 1337] if Nq == 1 else [3000, 4, 1337]
    q = rand((B, Nq, Hq, d), 11 + d + Nq, 2.0)
    k, v = caches(B, Nk, Hkv, d, lens, 12 + d)
    o, lse, n = run_decode(q, k, v, lens, causal, d ** -0.5)
    assert n > 0   # several splits: the merge kernel ran
    oo, lo = oracle.attn_decode_oracle(q, k, v, lens, causal, d ** -0.5)
    compare(o, lse, oo, lo, f"decode d={d} causal={causal} Nq={Nq}")


@pytest.mark.parametrize("Hq,Hkv,Nq", [(32, 8, 1), (16, 1, 8), (64, 1, 2), (4, 4, 32)])
def test_decode_group_shapes(Hq, Hkv, Nq):
    B, Nk, d = 2, 2500, 128
    lens = [2500, 999]
    q = rand((B, Nq, Hq, d), 21 + Hq + Nq)
    k, v = caches(B, Nk, Hkv, d, lens, 22)
    o, lse, _ = run_decode(q, k, v, lens, True, d ** -0.5)
    oo, lo = oracle.attn_decode_oracle(q, k, v, lens, True, d ** -0.5)
    compare(o, lse, oo, lo, f"decode Hq={Hq} Hkv={Hkv} Nq={Nq}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv,Nq", [(8, 4, 4), (4, 2, 2), (6, 2, 1), (3, 1, 2), (8, 8, 1)])
def test_decode_few_rows_per_kv_head(d, Hq, Hkv, Nq):
    """Group x Nq <= 8 rows per kv head (the CUDA-core kernel), causal, with
    several new positions and row counts that are not powers of two (the
    kernel pads to 1, 2, 4 or 8 rows); lengths that split the keys and
    lengths that do not."""
    B, Nk = 3, 2100
    lens = [2100, Nq, 777]
    q = rand((B, Nq, Hq, d), 101 + Hq + Nq + d, 2.0)
    k, v = caches(B, Nk, Hkv, d, lens, 102 + d)
    o, lse, _ = run_decode(q, k, v, lens, True, d ** -0.5)
    oo, lo = oracle.attn_decode_oracle(q, k, v, lens, True, d ** -0.5)
    compare(o, lse, oo, lo, f"decode d={d} Hq={Hq} Hkv={Hkv} Nq={Nq}")


def test_decode_few_rows_many_sequences():
    """Enough (sequence, kv head) pairs for one unit per CTA (no split),
    causal with two new positions, varied lengths."""
    B, Nq, Hq, Hkv, Nk, d = 48, 2, 8, 4, 700, 128
    lens = [Nq + (b * 37) % 690 for b in range(B)]
    q = rand((B, Nq, Hq, d), 111, 2.0)
    k, v = caches(B, Nk, Hkv, d, lens, 112)
    o, lse, n = run_decode(q, k, v, lens, True, d ** -0.5)
    assert n == 0
    oo, lo = oracle.attn_decode_oracle(q, k, v, lens, True, d ** -0.5)
    compare(o, lse, oo, lo, "decode few rows, many sequences")


def test_decode_single_split_writes_directly():
    """Enough (sequence, kv head) pairs for every SM: one split, no merge
    kernel and no workspace."""
    B, Nq, Hq, Hkv, Nk, d = 64, 1, 16, 8, 256, 64
    assert pkg.attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d) == 0
    lens = [256 - (b * 7) % 200 for b in range(B)]
    q = rand((B, Nq, Hq, d), 31)
    k, v = caches(B, Nk, Hkv, d, lens, 32)
    o, lse, n = run_decode(q, k, v, lens, False, d ** -0.5)
    assert n == 0
    oo, lo = oracle.attn_decode_oracle(q, k, v, lens, False, d ** -0.5)
    compare(o, lse, oo, lo, "decode single split")


def test_decode_full_caches_without_lengths():
    B, Nq, Hq, Hkv, Nk, d = 2, 2, 8, 8, 1500, 64
    q = rand((B, Nq, Hq, d), 41, 3.0)
    k, v = caches(B, Nk, Hkv, d, [Nk] * B, 42)
    o, lse, _ = run_decode(q, k, v, None, True, d ** -0.5)
    oo, lo = oracle.attn_decode_oracle(q, k, v, [Nk] * B, True, d ** -0.5)
    compare(o, lse, oo, lo, "decode without seqlens")


def test_decode_matches_prefill_rows():
    """The decode of the last Nq positions equals the last Nq rows of the
    causal prefill kernel over the whole sequence."""
    N, Nq, Hq, Hkv, d = 1024, 3, 8, 2, 128
    q = rand((1, N, Hq, d), 51)
    k = rand((1, N, Hkv, d), 52)
    v = rand((1, N, Hkv, d), 53)
    dev = torch.device("cuda:0")
    of, lf = pkg.attention(q.to(dev), k.to(dev), v.to(dev), causal=True)
    o, lse, _ = run_decode(q[:, N - Nq:].contiguous(), k, v, [N], True, d ** -0.5)
    assert np.abs(o[0] - of[0, N - Nq:].float().cpu().numpy()).max() <= 2e-2
    assert np.abs(lse[0] - lf[0, :, N - Nq:].cpu().numpy()).max() <= 1e-3


def test_decode_bad_lengths_reported():
    B, Nq, Hq, Hkv, Nk, d = 2, 2, 4, 2, 600, 64
    q = rand((B, Nq, Hq, d), 61)
    k, v = caches(B, Nk, Hkv, d, [600, 600], 62)
    o, lse, _ = run_decode(q, k, v, [600, 1], False, d ** -0.5, check_status=False)
    assert pkg.attn_get_status() == pkg.ATTN_OK   # the run above read and cleared it
    o, lse, _ = run_decode(q, k, v, [601, 300], False, d ** -0.5, check_status=False)
    # sequence 0 is out of range: its rows stay unwritten, sequence 1 is right
    assert np.isnan(o[0]).all() and np.isnan(lse[0]).all()
    oo, lo = oracle.attn_decode_oracle(q[1:], k[1:], v[1:], [300], False, d ** -0.5)
    compare(o[1:], lse[1:], oo, lo, "decode good sequence next to a bad one")


def test_decode_bad_length_sets_status():
    B, Nq, Hq, Hkv, Nk, d = 1, 2, 4, 2, 600, 64
    q = rand((B, Nq, Hq, d), 71)
    k, v = caches(B, Nk, Hkv, d, [600], 72)
    dev = torch.device("cuda:0")
    o = torch.empty((B, Nq, Hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    ws = torch.empty((1 << 20,), dtype=torch.float32, device=dev)
    sl = torch.tensor([1], dtype=torch.int32, device=dev)   # fewer keys than queries
    pkg.attn_fwd_decode(q.to(dev), k.to(dev), v.to(dev), o, lse, B, Hq, Hkv, Nq, Nk, d, 0.125,
                        False, sl, ws)
    assert pkg.attn_get_status() == pkg.ATTN_ERR_BAD_SEQLENS


def test_decode_small_workspace_rejected():
    B, Nq, Hq, Hkv, Nk, d = 1, 1, 8, 8, 8192, 128
    n = pkg.attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d)
    assert n > 0
    dev = torch.device("cuda:0")
    q = torch.zeros((B, Nq, Hq, d), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((B, Nk, Hkv, d), dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    ws = torch.empty((n // 4 - 4,), dtype=torch.float32, device=dev)
    rc = pkg.attn_fwd_decode(q, k, k, o, lse, B, Hq, Hkv, Nq, Nk, d, 0.1, False, None, ws,
                             check=False)
    assert rc == pkg.ATTN_ERR_INVALID_ARG
