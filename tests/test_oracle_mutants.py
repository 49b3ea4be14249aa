"""The oracle's pins must catch plausible slips.

Each case compiles a copy of the oracle with one deliberate mistake (on the
CPU, in a temporary directory) and checks that at least one pin from
``test_oracle.py`` rejects it.  This guards the pins themselves: a pin set
that a wrong oracle passes would prove nothing.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from test_oracle import brute_force, rand_bf16

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "causal bound off by one": ("int64_t jhi = causal ? pos :", "int64_t jhi = causal ? pos - 1 :"),
    "decode offset dropped": ("const int64_t pos = i + k_len[s] - q_len[s];",
                              "const int64_t pos = i;"),
    "group mapping h % Hkv": ("int kv = h / group;", "int kv = h % Hkv;"),
    "log2 instead of ln": ("*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    "scale dropped": ("double sc = scale * acc;", "double sc = acc;"),
    "value row fixed": ("const uint16_t *vrow = vbase + (jlo + n) * kstride;",
                        "const uint16_t *vrow = vbase;"),
    "key used as value": ("out[t] += pw * bf16_to_double(vrow[t]);",
                          "out[t] += pw * bf16_to_double(kbase[(jlo + n) * kstride + t]);"),
    "no max subtraction": ("double p = exp(scores[n] - m);", "double p = exp(scores[n]);"),
    "max starts at zero": ("double m = scores[0];", "double m = 0.0;"),
    "no normalisation": ("for (int t = 0; t < d; ++t) out[t] /= l;", ""),
    "window lower bound off by one": ("(wl >= 0 && pos - wl > 0) ? pos - wl : 0",
                                      "(wl >= 0 && pos - wl + 1 > 0) ? pos - wl + 1 : 0"),
    "window right bound ignored": ("if (!causal && wr >= 0 && pos + wr < jhi) jhi = pos + wr;", ""),
    "alibi sign": ("sc -= slope *", "sc += slope *"),
    "alibi distance one-sided": ("(double)(i > j ? i - j : j - i)", "(double)(i - j)"),
    "soft cap not scaled back": ("sc = cap * tanh(sc / cap);", "sc = tanh(sc / cap);"),
    "soft cap on the raw product": ("double sc = scale * acc;\n    if (cap > 0.0) sc = cap * tanh(sc / cap);",
                                    "double sc = acc;\n    if (cap > 0.0) sc = cap * tanh(sc / cap);\n    sc *= scale;"),
    "backward: D with the wrong sign": ("const double ds = p[j] * (dp[j] - D);",
                                        "const double ds = p[j] * (dp[j] + D);"),
    "backward: dK without the scale": ("dkj[t] += scale * ds * bf16_to_double(qi[t]);",
                                       "dkj[t] += ds * bf16_to_double(qi[t]);"),
    "backward: dV weighted by dS": ("dvj[t] += p[j] * bf16_to_double(doi[t]);",
                                    "dvj[t] += ds * bf16_to_double(doi[t]);"),
    "backward: causal bound off by one": ("const int64_t n = causal ? i + 1 : L;",
                                          "const int64_t n = causal ? i : L;"),
    "backward: P not normalised": ("      p[j] /= l;\n", ""),
    "bf16 rounding truncates": ("ldexp(rint(ldexp(ax, -spacing_exp)), spacing_exp)",
                                "ldexp(floor(ldexp(ax, -spacing_exp)), spacing_exp)"),
    "bf16 rounding ties upward": ("ldexp(rint(ldexp(ax, -spacing_exp)), spacing_exp)",
                                  "ldexp(floor(ldexp(ax, -spacing_exp) + 0.5), spacing_exp)"),
    "bf16 rounding through float first": ("const double ax = fabs(x);",
                                          "const double ax = (double)(float)fabs(x);"),
    "bf16 spacing one bit too fine": ("int spacing_exp = (e - 1) - 7;",
                                      "int spacing_exp = (e - 1) - 8;"),
    "q row of the kv head": ("const uint16_t *qrow = q + (q_start[s] + i) * qstride + (int64_t)h * d;",
                             "const uint16_t *qrow = q + (q_start[s] + i) * qstride + (int64_t)kv * d;"),
}


def _build_mutant(tmp_path, before, after):
    src = open(SRC).read()
    assert src.count(before) == 1, before
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(before, after))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                    "-o", str(so), str(path), "-lm"], check=True)
    return oracle.load_library(str(so))


def _pins_pass(lib) -> bool:
    """A compact run of the pins; False as soon as one fails."""
    # brute force, GQA, causal and not, packed sequences
    for causal in (False, True):
        lens = [7, 3, 9]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T, Hq, Hkv, d = int(cu[-1]), 4, 2, 5
        q = rand_bf16((T, Hq, d), 1, 2.0)
        k = rand_bf16((T, Hkv, d), 2)
        v = rand_bf16((T, Hkv, d), 3)
        o, lse = oracle.attn_fwd_oracle(q, k, v, 3, Hq, Hkv, T, d, 0.5, causal,
                                        cu_seqlens=cu, lib=lib)
        Ob, Lb = brute_force(q, k, v, lens, Hq, Hkv, d, 0.5, causal)
        if not (np.allclose(o, Ob, atol=1e-12, rtol=0) and np.allclose(lse, Lb.T, atol=1e-12, rtol=0)):
            return False
    # large scores stay finite and match the library log-sum-exp
    q = rand_bf16((1, 64, 2, 16), 81, 30.0)
    k = rand_bf16((1, 64, 2, 16), 82, 30.0)
    v = rand_bf16((1, 64, 2, 16), 83)
    o, lse = oracle.attn_fwd_oracle(q, k, v, 1, 2, 2, 64, 16, 1.0, False, lib=lib)
    S = torch.einsum("bihd,bjhd->bhij", q.double(), k.double())
    if not (np.isfinite(o).all() and np.allclose(lse, torch.logsumexp(S, -1).numpy(), rtol=1e-13)):
        return False
    # score and mask variants against the exact-summation evaluation
    from test_oracle import VARIANTS, brute_force_var
    lens = [7, 3, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, Hq, Hkv, d = int(cu[-1]), 4, 2, 5
    q = rand_bf16((T, Hq, d), 11, 2.0)
    k = rand_bf16((T, Hkv, d), 12)
    v = rand_bf16((T, Hkv, d), 13)
    for var in VARIANTS:
        slopes = [0.5 ** (h + 1) for h in range(Hq)] if var.get("slopes") else None
        window, cap = var.get("window", (-1, -1)), var.get("cap", 0.0)
        o, lse = oracle.attn_fwd_oracle(q, k, v, 3, Hq, Hkv, T, d, 0.6, var["causal"],
                                        cu_seqlens=cu, window=window, softcap=cap,
                                        alibi_slopes=slopes, lib=lib)
        Ob, Lb = brute_force_var(q, k, v, lens, Hq, Hkv, d, 0.6, var["causal"], window, cap,
                                 slopes)
        if not (np.allclose(o, Ob, atol=1e-12, rtol=0) and np.allclose(lse, Lb.T, atol=1e-12, rtol=0)):
            return False
    # decode shapes: a few queries at the end of longer key sequences
    from test_oracle import brute_force_decode
    for causal in (False, True):
        B, Nq, Nk, Hq, Hkv, d = 2, 3, 11, 4, 2, 5
        kl = [11, 6]
        q = rand_bf16((B, Nq, Hq, d), 61, 2.0)
        k = rand_bf16((B, Nk, Hkv, d), 62)
        v = rand_bf16((B, Nk, Hkv, d), 63)
        o, lse = oracle.attn_decode_oracle(q, k, v, kl, causal, 0.6, lib=lib)
        Ob, Lb = brute_force_decode(q, k, v, kl, causal, 0.6)
        if not (np.allclose(o, Ob, atol=1e-12, rtol=0) and np.allclose(lse, Lb, atol=1e-12, rtol=0)):
            return False
    # backward against torch fp64 autograd
    for causal in (False, True):
        B, N, Hq, Hkv, d, scale = 1, 9, 4, 2, 6, 0.45
        q = rand_bf16((B, N, Hq, d), 131, 2.0)
        k = rand_bf16((B, N, Hkv, d), 132)
        v = rand_bf16((B, N, Hkv, d), 133)
        g = rand_bf16((B, N, Hq, d), 134)
        dq, dk, dv = oracle.attn_bwd_oracle(q, k, v, g, B, Hq, Hkv, N, d, scale, causal, lib=lib)
        qt, kt, vt = (x.double().requires_grad_() for x in (q, k, v))
        s_ = torch.einsum("bihd,bjhd->bhij", qt, kt.repeat_interleave(2, dim=2)) * scale
        if causal:
            s_ = s_.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
        o = torch.einsum("bhij,bjhd->bihd", torch.softmax(s_, -1), vt.repeat_interleave(2, dim=2))
        o.backward(g.double())
        for mine, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
            if not np.allclose(mine, ref.numpy(), atol=1e-12, rtol=0):
                return False
    # the round_p diagnostic's rounding to bf16
    from test_oracle import round_bf16_pins_hold
    if not round_bf16_pins_hold(lib):
        return False
    # Q = 0 closed form
    q = torch.zeros((1, 9, 2, 4), dtype=torch.bfloat16)
    k = rand_bf16((1, 9, 2, 4), 5)
    o, lse = oracle.attn_fwd_oracle(q, k, k, 1, 2, 2, 9, 4, 1.0, True, lib=lib)
    if not all(abs(lse[0, h, i] - math.log(i + 1)) < 1e-14 for h in range(2) for i in range(9)):
        return False
    return True


def test_unmutated_oracle_passes_compact_pins():
    assert _pins_pass(oracle._load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    lib = _build_mutant(tmp_path, before, after)
    assert not _pins_pass(lib), f"pins did not catch: {name}"
