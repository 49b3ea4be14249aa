"""Parity of the score and mask variants (key window with tile skipping, soft
cap, ALiBi; tang, section 7.3) with the fp64 oracle, through attn_fwd_ex.

Same tolerances and NaN-filled, guarded outputs as test_attn_gpu.py.
"""
import math
import time

import numpy as np
import pytest
import torch

import oracle
import tensor_program_compilers_gb300 as pkg
from test_attn_gpu import Run, compare, rand

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg.build()
    torch.cuda.set_device(0)
    pkg.attn_get_status()


class RunEx(Run):
    """Run with window / soft cap / ALiBi slopes."""

    def __init__(self, *args, window=None, softcap=0.0, slopes=None, **kw):
        super().__init__(*args, **kw)
        self.window, self.softcap = window, softcap
        self.slopes = None if slopes is None else torch.tensor(slopes, dtype=torch.float32,
                                                               device="cuda:0")

    def __call__(self, check_status=True):
        B, Hq, Hkv, N, d, scale, causal = self.args
        rc = pkg.attn_fwd_ex(self.q, self.k, self.v, self.o, self.lse, B, Hq, Hkv, N, d, scale,
                             causal, self.cu, window=self.window, softcap=self.softcap,
                             alibi_slopes=self.slopes, check=False)
        assert rc == pkg.ATTN_OK, pkg.attn_status_string(rc)
        st = pkg.attn_get_status()
        if check_status:
            assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
        assert (self.obuf[:4096] == 7.0).all() and (self.obuf[-4096:] == 7.0).all()
        assert (self.lbuf[:4096] == 7.0).all() and (self.lbuf[-4096:] == 7.0).all()
        return self.o.float().cpu().numpy(), self.lse.cpu().numpy()


def alibi_slopes(H):
    """The usual geometric slopes 2^(-8 (h + 1) / H)."""
    return [2.0 ** (-8.0 * (h + 1) / H) for h in range(H)]


def check_fixed(B, Hq, Hkv, N, d, causal, seed, qmult=1.0, window=None, softcap=0.0,
                slopes=None):
    q = rand((B, N, Hq, d), seed, qmult)
    k = rand((B, N, Hkv, d), seed + 1)
    v = rand((B, N, Hkv, d), seed + 2)
    scale = d ** -0.5
    o, lse = RunEx(q, k, v, B, Hq, Hkv, N, d, scale, causal, window=window, softcap=softcap,
                   slopes=slopes)()
    oo, lo = oracle.attn_fwd_oracle(q, k, v, B, Hq, Hkv, N, d, scale, causal,
                                    window=(-1, -1) if window is None else window,
                                    softcap=softcap, alibi_slopes=slopes)
    return compare(o, lse.reshape(B, Hq, N), oo, lo,
                   f"d={d} N={N} causal={causal} window={window} cap={softcap} "
                   f"alibi={slopes is not None}")


# ----------------------------------------------------------------- key windows
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("window", [(127, -1), (0, 0), (200, -1), (1000, 5)])
def test_causal_window(d, window):
    check_fixed(1, 4, 2, 700, d, True, 100 + d, window=window)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("window", [(64, 64), (0, 300), (300, 0), (5, 129)])
def test_bidirectional_window(d, window):
    check_fixed(2, 2, 1, 555, d, False, 200 + d, window=window)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_packed_window(d):
    lens = [1, 127, 300, 0, 700, 129]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, Hq, Hkv = int(cu[-1]), 4, 2
    q = rand((T, Hq, d), 301 + d, 2.0)
    k = rand((T, Hkv, d), 302 + d)
    v = rand((T, Hkv, d), 303 + d)
    for causal, window in ((True, (127, -1)), (False, (100, 40))):
        o, lse = RunEx(q, k, v, len(lens), Hq, Hkv, T, d, d ** -0.5, causal, cu=cu,
                       window=window)()
        oo, lo = oracle.attn_fwd_oracle(q, k, v, len(lens), Hq, Hkv, T, d, d ** -0.5, causal,
                                        cu_seqlens=cu, window=window)
        compare(o, lse.reshape(Hq, T), oo, lo, f"packed d={d} causal={causal} window={window}")


# ----------------------------------------------------------------- score modifiers
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("cap", [5.0, 30.0])
def test_softcap(d, causal, cap):
    check_fixed(1, 4, 2, 400, d, causal, 400 + d, qmult=4.0, softcap=cap)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_alibi(d, causal):
    check_fixed(2, 4, 2, 333, d, causal, 500 + d, slopes=alibi_slopes(4))


@pytest.mark.parametrize("d", [64, 128])
def test_all_variants_together(d):
    check_fixed(1, 8, 2, 650, d, True, 600 + d, qmult=3.0, window=(250, -1), softcap=20.0,
                slopes=alibi_slopes(8))
    check_fixed(1, 8, 2, 650, d, False, 610 + d, qmult=3.0, window=(90, 170), softcap=8.0,
                slopes=alibi_slopes(8))


def test_alibi_zero_q_closed_form():
    """Q = 0: the weights of row i are exp(-slope |i - j|) (a geometric
    series), so LSE_i has a closed form."""
    B, N, H, d = 1, 300, 2, 64
    q = torch.zeros((B, N, H, d), dtype=torch.bfloat16)
    k = rand((B, N, H, d), 701)
    v = rand((B, N, H, d), 702)
    slopes = [0.05, 0.5]
    o, lse = RunEx(q, k, v, B, H, H, N, d, d ** -0.5, True, slopes=slopes)()
    lse = lse.reshape(B, H, N)
    for h, a in enumerate(slopes):
        r = math.exp(-a)
        ref = np.log((1 - r ** (np.arange(N) + 1)) / (1 - r))
        np.testing.assert_allclose(lse[0, h], ref, atol=1e-3, rtol=0)


# ----------------------------------------------------------------- tile skipping
def test_sliding_window_skips_key_tiles():
    """A causal window of 128 keys visits at most two key tiles per query
    tile, so at N = 16384 it must run far faster than full causal attention
    (which visits 64.5 on average), instead of computing masked tiles."""
    B, N, H, d = 1, 16384, 16, 64
    dev = torch.device("cuda:0")
    q = rand((B, N, H, d), 801).to(dev)
    k = rand((B, N, H, d), 802).to(dev)
    v = rand((B, N, H, d), 803).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)

    def timed(window):
        for _ in range(3):
            pkg.attn_fwd_ex(q, k, v, o, lse, B, H, H, N, d, d ** -0.5, True, window=window)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(10):
            pkg.attn_fwd_ex(q, k, v, o, lse, B, H, H, N, d, d ** -0.5, True, window=window)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / 10

    full, win = timed(None), timed((127, -1))
    assert pkg.attn_get_status() == pkg.ATTN_OK
    assert win < 0.2 * full, f"window {win * 1e3:.3f} ms vs causal {full * 1e3:.3f} ms"
