"""Parity of the paged-cache decode (attn_fwd_decode_paged: key/value rows
gathered page by page through a block table) with the fp64 oracle, through
the C ABI.  Same tolerances as test_attn_gpu.py."""
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


def paged_problem(B, Nq, Hq, Hkv, d, P, lens, seed, spare=7):
    """A pool with the sequences' pages in shuffled slots, unused slots full of
    NaN (any read of them would show), rows past a length inside a
    sequence's last page finite; table entries past the last page are -1."""
    max_blocks = max((L + P - 1) // P for L in lens) + 1
    need = sum((L + P - 1) // P for L in lens)
    num_pages = need + spare
    rng = np.random.default_rng(seed)
    slots = rng.permutation(num_pages)
    kc = torch.full((num_pages, P, Hkv, d), float("nan")).to(torch.bfloat16)
    vc = torch.full((num_pages, P, Hkv, d), float("nan")).to(torch.bfloat16)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    n = 0
    for b, L in enumerate(lens):
        for blk in range((L + P - 1) // P):
            s = int(slots[n]); n += 1
            table[b, blk] = s
            kc[s] = rand((P, Hkv, d), seed * 1000 + 2 * n)
            vc[s] = rand((P, Hkv, d), seed * 1000 + 2 * n + 1)
    q = rand((B, Nq, Hq, d), seed + 5, 2.0)
    return q, kc, vc, table, max_blocks, num_pages


def run_paged(q, kc, vc, table, max_blocks, num_pages, P, lens, causal, check_status=True):
    B, Nq, Hq, d = q.shape
    Hkv = kc.shape[2]
    dev = torch.device("cuda:0")
    dq, dk, dv = q.to(dev), kc.to(dev), vc.to(dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    tb = torch.tensor(table, dtype=torch.int32, device=dev)
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device=dev)
    n = pkg.attn_decode_paged_workspace_bytes(B, Hq, Hkv, Nq, max_blocks, P, d)
    ws = torch.empty(((max(n, 16) + 15) // 16 * 4,), dtype=torch.float32, device=dev)
    rc = pkg.attn_fwd_decode_paged(dq, dk, dv, o, lse, B, Hq, Hkv, Nq, d, d ** -0.5, causal, sl,
                                   tb, max_blocks, P, num_pages, ws, check=False)
    assert rc == pkg.ATTN_OK, pkg.attn_status_string(rc)
    st = pkg.attn_get_status()
    if check_status:
        assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    return o.float().cpu().numpy(), lse.cpu().numpy(), st


@pytest.mark.parametrize("P", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("d", [64, 128])
def test_paged_parity_page_sizes(P, d):
    B, Nq, Hq, Hkv = 3, 1, 8, 2
    lens = [1500, 1, 700]
    q, kc, vc, table, mb, npg = paged_problem(B, Nq, Hq, Hkv, d, P, lens, 10 + P + d)
    o, lse, _ = run_paged(q, kc, vc, table, mb, npg, P, lens, False)
    oo, lo = oracle.attn_decode_paged_oracle(q, kc, vc, lens, table, P, False, d ** -0.5)
    compare(o, lse, oo, lo, f"paged P={P} d={d}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_paged_parity_heads_and_queries(d, causal):
    B, Nq, Hq, Hkv, P = 2, 3, 16, 4, 64
    lens = [2000, 333]
    q, kc, vc, table, mb, npg = paged_problem(B, Nq, Hq, Hkv, d, P, lens, 50 + d)
    o, lse, _ = run_paged(q, kc, vc, table, mb, npg, P, lens, causal)
    oo, lo = oracle.attn_decode_paged_oracle(q, kc, vc, lens, table, P, causal, d ** -0.5)
    compare(o, lse, oo, lo, f"paged d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("P", [16, 64, 128])
def test_paged_few_rows_causal(d, P):
    """The CUDA-core kernel over pages: group 2 x Nq 3 = 6 rows per kv
    head, causal."""
    B, Nq, Hq, Hkv = 2, 3, 8, 4
    lens = [1333, 300]
    q, kc, vc, table, mb, npg = paged_problem(B, Nq, Hq, Hkv, d, P, lens, 60 + P + d)
    o, lse, _ = run_paged(q, kc, vc, table, mb, npg, P, lens, True)
    oo, lo = oracle.attn_decode_paged_oracle(q, kc, vc, lens, table, P, True, d ** -0.5)
    compare(o, lse, oo, lo, f"paged few rows P={P} d={d}")


def test_paged_page_size_not_a_power_of_two():
    """384-row pages (a multiple of 128, not a power of two: the page index
    is a division there)."""
    B, Nq, Hq, Hkv, d, P = 2, 1, 8, 2, 128, 384
    lens = [2000, 385]
    q, kc, vc, table, mb, npg = paged_problem(B, Nq, Hq, Hkv, d, P, lens, 77)
    o, lse, _ = run_paged(q, kc, vc, table, mb, npg, P, lens, False)
    oo, lo = oracle.attn_decode_paged_oracle(q, kc, vc, lens, table, P, False, d ** -0.5)
    compare(o, lse, oo, lo, "paged P=384")


def test_paged_matches_contiguous_decode():
    """Pages laid out in order are the contiguous caches: the two entry
    points give the same bits."""
    B, Nq, Hq, Hkv, d, P, nb = 2, 1, 8, 2, 128, 32, 40
    lens = [1280, 901]
    dev = torch.device("cuda:0")
    q = rand((B, Nq, Hq, d), 71).to(dev)
    k = rand((B, nb * P, Hkv, d), 72).to(dev)
    v = rand((B, nb * P, Hkv, d), 73).to(dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    table = torch.arange(B * nb, dtype=torch.int32, device=dev).reshape(B, nb)
    o1, l1 = pkg.decode(q, k, v, causal=False, seqlens_k=sl)
    o2 = torch.empty_like(o1)
    l2 = torch.empty_like(l1)
    n = pkg.attn_decode_paged_workspace_bytes(B, Hq, Hkv, Nq, nb, P, d)
    ws = torch.empty(((max(n, 16) + 15) // 16 * 4,), dtype=torch.float32, device=dev)
    pkg.attn_fwd_decode_paged(q, k.view(B * nb, P, Hkv, d), v.view(B * nb, P, Hkv, d), o2, l2,
                              B, Hq, Hkv, Nq, d, d ** -0.5, False, sl, table, nb, P, B * nb, ws)
    assert pkg.attn_get_status() == pkg.ATTN_OK
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_paged_bad_page_number_reported():
    B, Nq, Hq, Hkv, d, P = 1, 1, 4, 1, 64, 64
    lens = [300]
    q, kc, vc, table, mb, npg = paged_problem(B, Nq, Hq, Hkv, d, P, lens, 90, spare=0)
    table = table.copy()
    table[0, 1] = npg + 3   # outside the pool
    run_paged(q, kc, vc, table, mb, npg, P, lens, False, check_status=False)
    # run_paged read (and cleared) the status; run again and read it here
    dev = torch.device("cuda:0")
    o = torch.empty((B, Nq, Hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    ws = torch.empty((1 << 18,), dtype=torch.float32, device=dev)
    pkg.attn_fwd_decode_paged(q.to(dev), kc.to(dev), vc.to(dev), o, lse, B, Hq, Hkv, Nq, d, 0.125,
                              False, torch.tensor(lens, dtype=torch.int32, device=dev),
                              torch.tensor(table, device=dev), mb, P, npg, ws)
    assert pkg.attn_get_status() == pkg.ATTN_ERR_BAD_PAGE_TABLE
