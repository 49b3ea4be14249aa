"""fp64 CPU attention oracle -- TEST INFRASTRUCTURE ONLY.

This package checks the CUDA path; the library never imports it.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg use it.

``attn_fwd_oracle`` computes the plain two-pass definition of attention with a
causal mask, grouped-query heads and packed variable-length sequences, in fp64,
from the exact bf16 input values (see ``attn_oracle.c`` for the definition and
the passages it follows: tang, sections 2.1-2.4 and 6; TileLang explainer,
"FlashAttention, in tiles").  Optional score and mask variants (tang, section
7.3): a key window around each row, a soft cap and ALiBi slopes.

Parity status: pinned.  The tests in ``tests/test_oracle.py`` check it against
closed forms, invariants, an independent brute-force evaluation and the
online-softmax merge of chunk states.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` with gcc and OpenMP."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = [
            "gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
            "-o", _LIB, _SRC, "-lm",
        ]
        subprocess.run(cmd, check=True, timeout=300)
    return _LIB


def load_library(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_attn_fwd.restype = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # q k v
        ctypes.c_void_p, ctypes.c_void_p,                   # o lse
        ctypes.c_int, i64p, i64p, i64p, i64p,               # nseq, starts/lens
        ctypes.c_int, ctypes.c_int, ctypes.c_int,           # Hq Hkv d
        ctypes.c_double, ctypes.c_int, ctypes.c_int,        # scale causal round_p
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,      # nsel sel nthreads
    ]
    lib.oracle_attn_fwd_var.restype = ctypes.c_int
    lib.oracle_attn_fwd_var.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # q k v
        ctypes.c_void_p, ctypes.c_void_p,                   # o lse
        ctypes.c_int, i64p, i64p, i64p, i64p,               # nseq, starts/lens
        ctypes.c_int, ctypes.c_int, ctypes.c_int,           # Hq Hkv d
        ctypes.c_double, ctypes.c_int,                      # scale causal
        ctypes.c_int64, ctypes.c_int64, ctypes.c_double,    # wl wr cap
        ctypes.c_void_p, ctypes.c_int,                      # slopes round_p
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,      # nsel sel nthreads
    ]
    lib.oracle_attn_bwd.restype = ctypes.c_int
    lib.oracle_attn_bwd.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # q k v dout
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,                   # dq dk dv
        ctypes.c_int, i64p, i64p,                                            # nseq start len
        ctypes.c_int, ctypes.c_int, ctypes.c_int,                            # Hq Hkv d
        ctypes.c_double, ctypes.c_int, ctypes.c_int,                         # scale causal nthreads
    ]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_round_bf16.restype = None
    lib.oracle_round_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = load_library(_LIB)
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def round_bf16(x, lib=None) -> np.ndarray:
    """The oracle's rounding of doubles to the nearest bf16 value (ties to
    even), as used by the ``round_p`` diagnostic; returned as float64."""
    lib = lib or _load()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty_like(a)
    lib.oracle_round_bf16(a.ctypes.data, out.ctypes.data, a.size)
    return out


def _bits(x) -> np.ndarray:
    """bf16 tensor/array -> contiguous uint16 numpy array of its bits."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            assert x.dtype == torch.bfloat16, x.dtype
            return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    assert a.dtype == np.uint16, a.dtype
    return a


def attention_core(q, k, v, q_start, q_len, k_start, k_len, Hq, Hkv, d, scale,
                   causal, round_p=False, sel=None, nthreads=0, lib=None,
                   window=(-1, -1), softcap=0.0, alibi_slopes=None):
    """Direct call of the C oracle.

    q: bf16 [rows_q, Hq, d]; k, v: bf16 [rows_k, Hkv, d] (torch bf16 tensors
    or uint16 bit arrays).  Sequence s owns query rows q_start[s] ..
    q_start[s]+q_len[s]-1 and keys k_start[s] .. k_start[s]+k_len[s]-1.

    Returns (o, lse) in fp64: with sel=None, o is [rows_q, Hq, d] and lse
    [rows_q, Hq] (rows outside every sequence stay NaN); with sel an int32
    array of (s, h, i) triples, o is [n, d] and lse [n].

    Variants: window = (wl, wr) keeps keys i - wl <= j <= i + wr (negative:
    unbounded; causal implies wr = 0); softcap > 0 maps a scaled score s to
    softcap * tanh(s / softcap); alibi_slopes (Hq values) subtract
    slope[h] * |i - j| after the cap.
    """
    lib = _load() if lib is None else lib
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    rows_q = qb.size // (Hq * d)
    nseq = len(q_len)
    arr = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.int64))
    qs, ql, ks, kl = arr(q_start), arr(q_len), arr(k_start), arr(k_len)
    for s in range(nseq):
        assert qs[s] + ql[s] <= rows_q
        assert ks[s] + kl[s] <= kb.size // (Hkv * d)
    if sel is None:
        o = np.full((rows_q, Hq, d), np.nan)
        lse = np.full((rows_q, Hq), np.nan)
        nsel, selp = -1, None
    else:
        sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 3))
        o = np.full((sel.shape[0], d), np.nan)
        lse = np.full((sel.shape[0],), np.nan)
        nsel, selp = sel.shape[0], sel.ctypes.data
    i64 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    slopes = None
    if alibi_slopes is not None:
        slopes = np.ascontiguousarray(np.asarray(alibi_slopes, dtype=np.float64).reshape(-1))
        assert slopes.size == Hq
    wl, wr = (int(window[0]), int(window[1]))
    rc = lib.oracle_attn_fwd_var(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, o.ctypes.data, lse.ctypes.data,
        nseq, i64(qs), i64(ql), i64(ks), i64(kl), Hq, Hkv, d, float(scale),
        int(bool(causal)), wl, wr, float(softcap),
        None if slopes is None else slopes.ctypes.data, int(bool(round_p)), nsel, selp,
        int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd rejected its arguments (code {rc})")
    return o, lse


def attn_fwd_oracle(q, k, v, B, Hq, Hkv, N, d, scale, causal, cu_seqlens=None,
                    round_p=False, rows=None, nthreads=0, lib=None, window=(-1, -1),
                    softcap=0.0, alibi_slopes=None):
    """The oracle in the library's calling convention and layouts.

    Fixed batch (cu_seqlens None): q, o are [B, N, Hq, d]; k, v [B, N, Hkv, d];
    LSE is [B, Hq, N].  Packed (cu_seqlens = B+1 offsets): q, o [T, Hq, d];
    k, v [T, Hkv, d]; LSE [Hq, T], T = cu_seqlens[B].

    rows=None computes everything and returns (o, lse) in those layouts (fp64).
    rows = array of (seq, h, i) triples computes only those rows and returns
    (o [n, d], lse [n]).  window, softcap, alibi_slopes: see attention_core.
    """
    if cu_seqlens is None:
        starts = [b * N for b in range(B)]
        lens = [N] * B
        T = B * N
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64).reshape(-1)
        assert cu.size == B + 1
        starts = cu[:-1].tolist()
        lens = (cu[1:] - cu[:-1]).tolist()
        T = int(cu[-1])
    o, lse = attention_core(q, k, v, starts, lens, starts, lens, Hq, Hkv, d, scale,
                            causal, round_p=round_p, sel=rows, nthreads=nthreads,
                            lib=lib, window=window, softcap=softcap,
                            alibi_slopes=alibi_slopes)
    if rows is not None:
        return o, lse
    if cu_seqlens is None:
        o = o.reshape(B, N, Hq, d)
        lse = lse.reshape(B, N, Hq).transpose(0, 2, 1).copy()
    else:
        o = o.reshape(T, Hq, d)
        lse = lse.reshape(T, Hq).T.copy()
    return o, lse


def attn_decode_oracle(q, k, v, seqlens_k, causal, scale, nthreads=0, lib=None):
    """The oracle in the decode convention: q [B, Nq, Hq, d] are the last Nq
    positions of sequences whose keys are k, v [B, Nk_max, Hkv, d] rows
    0 .. seqlens_k[b] - 1 (the rest of each cache is ignored).  With causal,
    query r of sequence b sees keys j <= seqlens_k[b] - Nq + r.

    Returns (o [B, Nq, Hq, d], lse [B, Hq, Nq]) in fp64.
    """
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    kl = [int(x) for x in np.asarray(seqlens_k).reshape(-1)]
    assert len(kl) == B and all(Nq <= x <= Nk for x in kl)
    o, lse = attention_core(q.reshape(B * Nq, Hq, d), k.reshape(B * Nk, Hkv, d),
                            v.reshape(B * Nk, Hkv, d), [b * Nq for b in range(B)], [Nq] * B,
                            [b * Nk for b in range(B)], kl, Hq, Hkv, d, scale, causal,
                            nthreads=nthreads, lib=lib)
    return o.reshape(B, Nq, Hq, d), lse.reshape(B, Nq, Hq).transpose(0, 2, 1).copy()


def attn_decode_paged_oracle(q, k_cache, v_cache, seqlens_k, block_table, page_size, causal,
                             scale, nthreads=0, lib=None):
    """The decode oracle over paged caches (tang, section 2.1 "Views": a paged
    KV cache is a gathered read -- the page holding key j is data, read from
    the block table).  Key j of sequence b is row j % page_size of page
    block_table[b, j // page_size] of k_cache, v_cache [num_pages, page_size,
    Hkv, d]; the gathered rows form ordinary caches for attn_decode_oracle.
    """
    import torch
    table = torch.as_tensor(np.asarray(block_table), dtype=torch.long)
    B, max_blocks = table.shape
    Nk = max_blocks * page_size
    kl = [int(x) for x in np.asarray(seqlens_k).reshape(-1)]
    Hkv, d = k_cache.shape[2], k_cache.shape[3]
    k = torch.zeros((B, Nk, Hkv, d), dtype=k_cache.dtype)
    v = torch.zeros((B, Nk, Hkv, d), dtype=v_cache.dtype)
    for b in range(B):
        for j in range(kl[b]):
            page = int(table[b, j // page_size])
            k[b, j] = k_cache[page, j % page_size]
            v[b, j] = v_cache[page, j % page_size]
    return attn_decode_oracle(q, k, v, kl, causal, scale, nthreads=nthreads, lib=lib)


def attn_bwd_oracle(q, k, v, dout, B, Hq, Hkv, N, d, scale, causal, cu_seqlens=None, nthreads=0,
                    lib=None):
    """Gradients (dq, dk, dv) in fp64 of O = attention(q, k, v) against the
    output gradient dout, in the forward's layouts (fixed batch [B, N, H, d],
    packed [T, H, d] with cu_seqlens).  See oracle_attn_bwd in attn_oracle.c
    (tang, section 3 "Gradients are comprehensions")."""
    lib = _load() if lib is None else lib
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    if cu_seqlens is None:
        starts = np.arange(B, dtype=np.int64) * N
        lens = np.full(B, N, dtype=np.int64)
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64).reshape(-1)
        starts, lens = cu[:-1].copy(), (cu[1:] - cu[:-1]).copy()
    rows = qb.size // (Hq * d)
    dq = np.full((rows, Hq, d), np.nan)
    dk = np.full((rows, Hkv, d), np.nan)
    dv = np.full((rows, Hkv, d), np.nan)
    i64 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    rc = lib.oracle_attn_bwd(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, gb.ctypes.data,
                             dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, len(lens),
                             i64(starts), i64(lens), Hq, Hkv, d, float(scale), int(bool(causal)),
                             int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd rejected its arguments (code {rc})")
    shape = lambda a, H: a.reshape((B, N, H, d) if cu_seqlens is None else (rows, H, d))
    return shape(dq, Hq), shape(dk, Hkv), shape(dv, Hkv)
