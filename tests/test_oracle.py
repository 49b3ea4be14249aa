"""Pins for the fp64 oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics
fix: an exact brute-force evaluation, closed forms, invariants and the
online-softmax monoid merge (tang, section 2.2 and Table 1; section 6: online
softmax is a commutative semigroup equal to two-pass softmax, and softmax is
shift invariant).  A plausible slip in the oracle -- a dropped scale, a
wrong causal bound, a wrong group mapping, log2 for ln, a transposed
operand, a missing max subtraction -- fails at least one of them.
"""
import math
import random

import numpy as np
import pytest
import torch

import oracle
from oracle import attention_core, attn_fwd_oracle


def bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def rand_bf16(shape, seed, mult=1.0):
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * mult).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# (viii) brute force with exact summation, on tiny inputs
# ---------------------------------------------------------------------------
def brute_force(q, k, v, lens, Hq, Hkv, d, scale, causal):
    """Exact-summation evaluation straight from the softmax definition."""
    qf = q.float().tolist()
    kf = k.float().tolist()
    vf = v.float().tolist()
    g = Hq // Hkv
    T = sum(lens)
    O = [[[0.0] * d for _ in range(Hq)] for _ in range(T)]
    LSE = [[0.0] * Hq for _ in range(T)]
    start = 0
    for L in lens:
        for i in range(L):
            for h in range(Hq):
                kvh = h // g
                js = list(range(i + 1)) if causal else list(range(L))
                sc = [scale * math.fsum(qf[start + i][h][t] * kf[start + j][kvh][t]
                                        for t in range(d)) for j in js]
                m = max(sc)
                e = [math.exp(x - m) for x in sc]
                l = math.fsum(e)
                for t in range(d):
                    O[start + i][h][t] = math.fsum(e[n] * vf[start + j][kvh][t]
                                                   for n, j in enumerate(js)) / l
                LSE[start + i][h] = m + math.log(l)
        start += L
    return np.array(O), np.array(LSE)


def brute_force_var(q, k, v, lens, Hq, Hkv, d, scale, causal, window=(-1, -1), cap=0.0,
                    slopes=None):
    """Exact-summation evaluation of the score and mask variants: keys
    i - wl <= j <= i + wr (negative: unbounded; causal: wr = 0), soft cap
    cap * tanh(s / cap) of the scaled score, then minus slope[h] * |i - j|."""
    qf, kf, vf = q.float().tolist(), k.float().tolist(), v.float().tolist()
    g = Hq // Hkv
    wl, wr = window
    T = sum(lens)
    O = np.zeros((T, Hq, d))
    LSE = np.zeros((T, Hq))
    start = 0
    for L in lens:
        for i in range(L):
            for h in range(Hq):
                kvh = h // g
                js = [j for j in range(L)
                      if (j <= i if causal else (wr < 0 or j <= i + wr))
                      and (wl < 0 or j >= i - wl)]
                sc = []
                for j in js:
                    x = scale * math.fsum(qf[start + i][h][t] * kf[start + j][kvh][t]
                                          for t in range(d))
                    if cap > 0:
                        x = cap * math.tanh(x / cap)
                    if slopes is not None:
                        x -= slopes[h] * abs(i - j)
                    sc.append(x)
                m = max(sc)
                e = [math.exp(x - m) for x in sc]
                l = math.fsum(e)
                for t in range(d):
                    O[start + i, h, t] = math.fsum(e[n] * vf[start + j][kvh][t]
                                                   for n, j in enumerate(js)) / l
                LSE[start + i, h] = m + math.log(l)
        start += L
    return O, LSE


def brute_force_decode(q, k, v, seqlens_k, causal, scale):
    """Exact-summation evaluation for queries that are the last Nq positions
    of their sequences (q [B, Nq, Hq, d], k/v [B, Nk, Hkv, d])."""
    B, Nq, Hq, d = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    qf, kf, vf = q.float().tolist(), k.float().tolist(), v.float().tolist()
    O = np.zeros((B, Nq, Hq, d))
    LSE = np.zeros((B, Hq, Nq))
    for b in range(B):
        L = int(seqlens_k[b])
        for r in range(Nq):
            pos = L - Nq + r
            js = list(range(pos + 1)) if causal else list(range(L))
            for h in range(Hq):
                kvh = h // g
                sc = [scale * math.fsum(qf[b][r][h][t] * kf[b][j][kvh][t] for t in range(d))
                      for j in js]
                m = max(sc)
                e = [math.exp(x - m) for x in sc]
                l = math.fsum(e)
                for t in range(d):
                    O[b, r, h, t] = math.fsum(e[n] * vf[b][j][kvh][t] for n, j in enumerate(js)) / l
                LSE[b, h, r] = m + math.log(l)
    return O, LSE


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (6, 3), (4, 1)])
def test_brute_force_fixed_batch(causal, Hq, Hkv):
    B, N, d = 2, 9, 5
    q = rand_bf16((B, N, Hq, d), 1)
    k = rand_bf16((B, N, Hkv, d), 2)
    v = rand_bf16((B, N, Hkv, d), 3)
    scale = 0.37
    o, lse = attn_fwd_oracle(q, k, v, B, Hq, Hkv, N, d, scale, causal)
    Ob, Lb = brute_force(q.reshape(B * N, Hq, d), k.reshape(B * N, Hkv, d),
                         v.reshape(B * N, Hkv, d), [N] * B, Hq, Hkv, d, scale, causal)
    np.testing.assert_allclose(o.reshape(B * N, Hq, d), Ob, rtol=0, atol=1e-12)
    # oracle LSE layout is [B, Hq, N]
    np.testing.assert_allclose(lse.transpose(0, 2, 1).reshape(B * N, Hq), Lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_packed(causal):
    lens = [5, 1, 7, 3, 0, 4]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, Hq, Hkv, d = int(cu[-1]), 4, 2, 6
    q = rand_bf16((T, Hq, d), 11, 2.0)
    k = rand_bf16((T, Hkv, d), 12)
    v = rand_bf16((T, Hkv, d), 13)
    o, lse = attn_fwd_oracle(q, k, v, len(lens), Hq, Hkv, T, d, 0.5, causal, cu_seqlens=cu)
    Ob, Lb = brute_force(q, k, v, lens, Hq, Hkv, d, 0.5, causal)
    np.testing.assert_allclose(o, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, Lb.T, rtol=0, atol=1e-12)   # LSE is [Hq, T]


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
def test_hand_worked_example():
    """q=[1,0]; keys [1,0],[0,1],[1,1]; values [1,0],[0,1],[2,3]; scale 1.
    Scores 1,0,1; with x = e^-1 the weights are 1, x, 1 over 2+x, so
    O = (3/(2+x), (x+3)/(2+x)) and LSE = 1 + ln(2+x)."""
    q = bf16([[[1.0, 0.0]], [[0.0, 0.0]], [[0.0, 0.0]]])          # [3, 1, 2]; row 0 used
    k = bf16([[[1.0, 0.0]], [[0.0, 1.0]], [[1.0, 1.0]]])
    v = bf16([[[1.0, 0.0]], [[0.0, 1.0]], [[2.0, 3.0]]])
    o, lse = attn_fwd_oracle(q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), 1, 1, 1, 3, 2,
                             1.0, False)
    x = math.exp(-1.0)
    assert abs(o[0, 0, 0, 0] - 3 / (2 + x)) < 1e-15
    assert abs(o[0, 0, 0, 1] - (x + 3) / (2 + x)) < 1e-15
    assert abs(lse[0, 0, 0] - (1 + math.log(2 + x))) < 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_zero_q_closed_form(causal):
    """Q = 0: every visible score is 0, so LSE_i = ln |valid(i)| (natural log)
    and O_i is the plain mean of V over the visible keys."""
    B, N, Hq, Hkv, d = 2, 13, 4, 2, 8
    q = torch.zeros((B, N, Hq, d), dtype=torch.bfloat16)
    k = rand_bf16((B, N, Hkv, d), 21)
    v = rand_bf16((B, N, Hkv, d), 22)
    o, lse = attn_fwd_oracle(q, k, v, B, Hq, Hkv, N, d, 0.125, causal)
    vf = v.double().numpy()
    for b in range(B):
        for h in range(Hq):
            for i in range(N):
                n = i + 1 if causal else N
                assert abs(lse[b, h, i] - math.log(n)) < 1e-14
                mean = np.array([math.fsum(vf[b, :n, h // 2, t]) / n for t in range(d)])
                np.testing.assert_allclose(o[b, i, h], mean, rtol=0, atol=1e-14)


def test_causal_row0():
    """A causal row 0 sees only key 0: O[0] = V[0] and LSE[0] = scale*q0.k0."""
    B, N, Hq, Hkv, d = 3, 17, 6, 2, 16
    q = rand_bf16((B, N, Hq, d), 31)
    k = rand_bf16((B, N, Hkv, d), 32)
    v = rand_bf16((B, N, Hkv, d), 33)
    scale = 0.25
    o, lse = attn_fwd_oracle(q, k, v, B, Hq, Hkv, N, d, scale, True)
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_array_equal(o[b, 0, h], vd[b, 0, h // 3])
            s00 = scale * math.fsum(qd[b, 0, h] * kd[b, 0, h // 3])
            assert abs(lse[b, h, 0] - s00) < 1e-14


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(causal):
    """With V = identity (d = N, V[j] = e_j) the output row IS the softmax row:
    non-negative, zero on masked keys, summing to 1."""
    N = 16
    q = rand_bf16((1, N, 2, N), 41, 3.0)
    k = rand_bf16((1, N, 1, N), 42)
    v = torch.eye(N, dtype=torch.bfloat16).reshape(1, N, 1, N)
    o, _ = attn_fwd_oracle(q, k, v, 1, 2, 1, N, N, 0.3, causal)
    P = o[0]                       # [N, H, N]
    assert (P >= 0).all()
    np.testing.assert_allclose(P.sum(axis=-1), 1.0, rtol=0, atol=1e-14)
    if causal:
        for i in range(N):
            assert (P[i, :, i + 1:] == 0).all()
            assert (P[i, :, : i + 1] > 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v(causal):
    """V = c everywhere gives O = c (weights sum to 1)."""
    B, N, Hq, d = 2, 40, 4, 8
    q = rand_bf16((B, N, Hq, d), 51, 4.0)
    k = rand_bf16((B, N, Hq, d), 52)
    v = torch.full((B, N, Hq, d), 0.75, dtype=torch.bfloat16)
    o, _ = attn_fwd_oracle(q, k, v, B, Hq, Hq, N, d, 0.5, causal)
    np.testing.assert_allclose(o, 0.75, rtol=0, atol=1e-14)


def test_key_permutation_noncausal():
    """Non-causal attention is a sum over keys: permuting K and V rows together
    changes nothing (tang section 5: keys may be permuted because the reduction
    is commutative and associative)."""
    B, N, Hq, Hkv, d = 2, 33, 4, 4, 8
    q = rand_bf16((B, N, Hq, d), 61)
    k = rand_bf16((B, N, Hkv, d), 62)
    v = rand_bf16((B, N, Hkv, d), 63)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(64))
    o1, l1 = attn_fwd_oracle(q, k, v, B, Hq, Hkv, N, d, 0.4, False)
    o2, l2 = attn_fwd_oracle(q, k[:, perm], v[:, perm], B, Hq, Hkv, N, d, 0.4, False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_shift_invariance(causal):
    """Adding the same constant to every score of a row shifts LSE by it and
    leaves O alone.  A spare feature t0 with q=1 and k=c adds scale*c to all
    scores."""
    B, N, Hq, d = 1, 24, 2, 8
    q = rand_bf16((B, N, Hq, d), 71)
    k = rand_bf16((B, N, Hq, d), 72)
    v = rand_bf16((B, N, Hq, d), 73)
    q[..., 0] = 1.0
    k0 = k.clone()
    k0[..., 0] = 0.0
    kc = k.clone()
    kc[..., 0] = 6.5
    scale = 0.5
    oa, la = attn_fwd_oracle(q, k0, v, B, Hq, Hq, N, d, scale, causal)
    ob, lb = attn_fwd_oracle(q, kc, v, B, Hq, Hq, N, d, scale, causal)
    np.testing.assert_allclose(ob, oa, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lb - la, scale * 6.5, rtol=0, atol=1e-12)


def test_large_scores_stay_finite():
    """Scores in the hundreds overflow exp() unless the row max is subtracted.
    The result must be finite and agree with the library log-sum-exp."""
    B, N, Hq, d = 1, 64, 2, 16
    q = rand_bf16((B, N, Hq, d), 81, 30.0)
    k = rand_bf16((B, N, Hq, d), 82, 30.0)
    v = rand_bf16((B, N, Hq, d), 83)
    o, lse = attn_fwd_oracle(q, k, v, B, Hq, Hq, N, d, 1.0, False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    S = torch.einsum("bihd,bjhd->bhij", q.double(), k.double())
    assert S.abs().max() > 800           # exp would overflow without the max
    np.testing.assert_allclose(lse, torch.logsumexp(S, dim=-1).numpy(), rtol=1e-13, atol=1e-10)


# ---------------------------------------------------------------------------
# (i) merge of online-softmax chunk states in any order and tree shape
# ---------------------------------------------------------------------------
def combine(a, b):
    """The online-softmax monoid on (m, l, o) with o carried unnormalised:
    (tang, section 2.2 and Table 1 row "online softmax")."""
    m1, l1, o1 = a
    m2, l2, o2 = b
    m = max(m1, m2)
    w1, w2 = math.exp(m1 - m), math.exp(m2 - m)
    return (m, l1 * w1 + l2 * w2, o1 * w1 + o2 * w2)


@pytest.mark.parametrize("seed", range(6))
def test_merge_of_chunk_states_matches_two_pass(seed):
    rng = random.Random(seed)
    nq, nk, Hq, Hkv, d = 5, 37, 2, 1, 6
    q = rand_bf16((nq, Hq, d), 100 + seed, 2.0)
    k = rand_bf16((nk, Hkv, d), 200 + seed)
    v = rand_bf16((nk, Hkv, d), 300 + seed)
    scale = 0.45
    o_full, l_full = attention_core(q, k, v, [0], [nq], [0], [nk], Hq, Hkv, d, scale, False)
    # random chunking of the keys (chunks need not be contiguous)
    keys = list(range(nk))
    rng.shuffle(keys)
    cuts = sorted(rng.sample(range(1, nk), rng.randint(1, 8)))
    chunks = [keys[a:b] for a, b in zip([0] + cuts, cuts + [nk])]
    states = []
    for c in chunks:
        idx = torch.tensor(c)
        oc, lc = attention_core(q, k[idx], v[idx], [0], [nq], [0], [len(c)], Hq, Hkv, d,
                                scale, False)
        # a normalised chunk result (o, lse) is the state (lse, 1, o)
        states.append([[(lc[i, h], 1.0, oc[i, h].copy()) for h in range(Hq)]
                       for i in range(nq)])
    for i in range(nq):
        for h in range(Hq):
            items = [s[i][h] for s in states]
            # random merge tree: repeatedly merge two random neighbours or any pair
            while len(items) > 1:
                a = rng.randrange(len(items))
                b = rng.randrange(len(items) - 1)
                b = b + 1 if b >= a else b
                x, y = items[a], items[b]
                merged = combine(x, y) if rng.random() < 0.5 else combine(y, x)
                items = [it for n, it in enumerate(items) if n not in (a, b)] + [merged]
            m, l, o = items[0]
            np.testing.assert_allclose(o / l, o_full[i, h], rtol=0, atol=1e-13)
            assert abs((m + math.log(l)) - l_full[i, h]) < 1e-13


# ---------------------------------------------------------------------------
# (ix) library softmax cross-check, and the bf16-rounding diagnostic
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_softmax_fp64(causal):
    B, N, Hq, Hkv, d = 2, 70, 8, 2, 32
    q = rand_bf16((B, N, Hq, d), 91, 2.0)
    k = rand_bf16((B, N, Hkv, d), 92)
    v = rand_bf16((B, N, Hkv, d), 93)
    scale = d ** -0.5
    o, lse = attn_fwd_oracle(q, k, v, B, Hq, Hkv, N, d, scale, causal)
    kk = k.double().repeat_interleave(Hq // Hkv, dim=2)
    vv = v.double().repeat_interleave(Hq // Hkv, dim=2)
    S = torch.einsum("bihd,bjhd->bhij", q.double(), kk) * scale
    if causal:
        S = S.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    P = torch.softmax(S, dim=-1)
    O = torch.einsum("bhij,bjhd->bihd", P, vv)
    np.testing.assert_allclose(o, O.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(S, -1).numpy(), rtol=0, atol=1e-12)


def bf16_neighbours():
    """Every pair of adjacent positive finite bf16 values (a, b), as doubles,
    with whether a's significand is even.  bf16 bit patterns of one sign are
    ordered like the values they encode, so adjacent patterns are adjacent
    values; the pair (0x7F, 0x80) crosses from subnormals to normals and the
    pairs whose lower value ends in 0x7F cross into the next binade."""
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)           # up to the largest finite
    vals = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    return vals[:-1], vals[1:], (bits[:-1] & 1) == 0


def round_bf16_pins_hold(lib=None) -> bool:
    """Pins of the oracle's double -> bf16 rounding (round to nearest, ties to
    even), from the definition alone: bf16 values are fixed points; an exact
    midpoint goes to the neighbour with the even significand; a value a tiny
    step off the midpoint goes to the nearer neighbour (truncation, rounding
    half up, or rounding to float first all fail one of these); signs are
    symmetric; values below half the smallest subnormal round to zero."""
    a, b, a_even = bf16_neighbours()
    r = lambda x: oracle.round_bf16(x, lib=lib)
    ok = np.array_equal(r(a), a) and np.array_equal(r(b), b)
    mid = (a + b) / 2                                  # exact in double
    ok &= np.array_equal(r(mid), np.where(a_even, a, b))
    eps = (b - a) * 2.0 ** -30                         # far below float's resolution here
    ok &= np.array_equal(r(mid + eps), b) and np.array_equal(r(mid - eps), a)
    ok &= np.array_equal(r(-(mid + eps)), -b) and np.array_equal(r(-mid), -np.where(a_even, a, b))
    tiny = 2.0 ** -134                                 # half the smallest subnormal (a tie)
    ok &= np.array_equal(r([tiny, tiny * 0.99, tiny * 1.01, 0.0]), [0.0, 0.0, 2.0 ** -133, 0.0])
    return bool(ok)


def test_round_bf16_is_nearest_even():
    assert round_bf16_pins_hold()


def test_round_p_rounds_each_weight_to_nearest_bf16():
    """Through the round_p switch: a row that sees two keys with scores 0 and
    s < 0 and one-hot values gets o[1] = bf16(e^s) / (1 + e^s) (the sum keeps
    the unrounded weights).  The recovered weight must be a bf16 value no
    farther from e^s than either of its bf16 neighbours."""
    n = 64
    svals = -np.linspace(0.01, 9.0, n)                  # one row per head
    d = 8
    q = torch.zeros((1, 2, n, d), dtype=torch.bfloat16)
    q[..., 0] = 1.0
    k = torch.zeros((1, 2, n, d))
    k[0, 1, :, 0] = torch.tensor(svals)
    k = k.to(torch.bfloat16)
    s = k[0, 1, :, 0].double().numpy()                  # the scores as bf16 inputs give them
    v = torch.zeros((1, 2, n, d), dtype=torch.bfloat16)
    v[0, 0, :, 0] = 1.0
    v[0, 1, :, 1] = 1.0
    o, lse = attn_fwd_oracle(q, k, v, 1, n, n, 2, d, 1.0, False, round_p=True)
    p = np.exp(s)
    w = o[0, 1, :, 1] * (1.0 + p)                       # recovered rounded weight
    np.testing.assert_allclose(o[0, 1, :, 0] * (1.0 + p), 1.0, rtol=1e-15)   # bf16(1) = 1
    np.testing.assert_allclose(lse[0, :, 1], np.log1p(p), rtol=0, atol=1e-15)
    # o * (1 + p) recovers the weight up to a couple of double roundings
    wb = torch.tensor(w, dtype=torch.float64).to(torch.float32)
    c = wb.double().numpy()
    assert (np.abs(w - c) <= 1e-15 * c).all(), "not a float value"
    bits = wb.view(torch.int32)
    assert (bits & 0xFFFF).eq(0).all(), "not a bf16 value"
    up = ((bits + 0x10000).view(torch.float32)).double().numpy()
    down = ((bits - 0x10000).view(torch.float32)).double().numpy()
    err = np.abs(c - p)
    assert (err <= np.abs(up - p)).all() and (err <= np.abs(down - p)).all()
    assert (c != p).all()                               # the switch did round


def test_row_selection_matches_full():
    B, N, Hq, Hkv, d = 2, 50, 4, 2, 16
    q = rand_bf16((B, N, Hq, d), 111)
    k = rand_bf16((B, N, Hkv, d), 112)
    v = rand_bf16((B, N, Hkv, d), 113)
    o, lse = attn_fwd_oracle(q, k, v, B, Hq, Hkv, N, d, 0.3, True)
    rows = [(1, 3, 49), (0, 0, 0), (1, 2, 17)]
    os_, ls = attn_fwd_oracle(q, k, v, B, Hq, Hkv, N, d, 0.3, True, rows=rows)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(os_[n], o[b, i, h])
        assert ls[n] == lse[b, h, i]


def test_rejects_bad_arguments():
    q = rand_bf16((1, 4, 3, 8), 1)
    k = rand_bf16((1, 4, 2, 8), 2)
    with pytest.raises(ValueError):
        attn_fwd_oracle(q, k, k, 1, 3, 2, 4, 8, 1.0, False)   # Hq % Hkv != 0
    with pytest.raises(ValueError):   # causal needs equal query/key lengths
        attention_core(q.reshape(4, 3, 8), k.reshape(4, 2, 8)[:, :1].contiguous(),
                       k.reshape(4, 2, 8)[:, :1].contiguous(), [0], [4], [0], [3], 3, 1, 8,
                       1.0, True)


def test_threads_reported():
    assert oracle.max_threads() >= 1


def test_golden_regression_record():
    import json
    import os
    import sys
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    from make_golden import case
    meta, q, k, v = case()
    rec = json.load(open(os.path.join(here, "oracle_regression_small.json")))
    o, lse = attn_fwd_oracle(q, k, v, meta["B"], meta["Hq"], meta["Hkv"], meta["N"], meta["d"],
                             meta["scale"], meta["causal"])
    np.testing.assert_allclose(o.reshape(-1), rec["o"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse.reshape(-1), rec["lse"], rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------
# score and mask variants (tang, section 7.3: soft cap, ALiBi, sliding window)
# ---------------------------------------------------------------------------
VARIANTS = [
    dict(causal=True, window=(3, -1)),
    dict(causal=False, window=(2, 4)),
    dict(causal=False, window=(-1, 1)),
    dict(causal=True, cap=1.5),
    dict(causal=False, cap=0.7),
    dict(causal=True, slopes=True),
    dict(causal=False, slopes=True),
    dict(causal=True, window=(4, -1), cap=2.0, slopes=True),
    dict(causal=False, window=(1, 2), cap=3.0, slopes=True),
]


@pytest.mark.parametrize("var", VARIANTS, ids=lambda v: "-".join(f"{k}={v[k]}" for k in v))
def test_variants_brute_force(var):
    lens = [7, 3, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, Hq, Hkv, d = int(cu[-1]), 4, 2, 5
    q = rand_bf16((T, Hq, d), 11, 2.0)
    k = rand_bf16((T, Hkv, d), 12)
    v = rand_bf16((T, Hkv, d), 13)
    slopes = [0.5 ** (h + 1) for h in range(Hq)] if var.get("slopes") else None
    window = var.get("window", (-1, -1))
    cap = var.get("cap", 0.0)
    o, lse = attn_fwd_oracle(q, k, v, 3, Hq, Hkv, T, d, 0.6, var["causal"], cu_seqlens=cu,
                             window=window, softcap=cap, alibi_slopes=slopes)
    Ob, Lb = brute_force_var(q, k, v, lens, Hq, Hkv, d, 0.6, var["causal"], window, cap,
                             slopes)
    np.testing.assert_allclose(o, Ob, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, Lb.T, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_window_of_one_key_returns_own_value(causal):
    """Window (0, 0): each row sees only its own key, so O = V[i] and
    LSE = s_ii (closed form)."""
    B, N, H, d = 2, 11, 3, 8
    q = rand_bf16((B, N, H, d), 21)
    k = rand_bf16((B, N, H, d), 22)
    v = rand_bf16((B, N, H, d), 23)
    o, lse = attn_fwd_oracle(q, k, v, B, H, H, N, d, 0.3, causal, window=(0, 0))
    np.testing.assert_allclose(o, v.double().numpy(), atol=1e-15, rtol=0)
    s_ii = 0.3 * np.einsum("bnhd,bnhd->bhn", q.double().numpy(), k.double().numpy())
    np.testing.assert_allclose(lse, s_ii, atol=1e-13, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_unbounded_or_wide_window_is_plain(causal):
    B, N, H, d = 1, 13, 2, 4
    q = rand_bf16((B, N, H, d), 31, 2.0)
    k = rand_bf16((B, N, H, d), 32)
    v = rand_bf16((B, N, H, d), 33)
    o0, l0 = attn_fwd_oracle(q, k, v, B, H, H, N, d, 0.5, causal)
    for w in ((-1, -1), (N, N), (N - 1, -1), (-1, N - 1)):
        o, l = attn_fwd_oracle(q, k, v, B, H, H, N, d, 0.5, causal, window=w)
        np.testing.assert_array_equal(o, o0)
        np.testing.assert_array_equal(l, l0)


@pytest.mark.parametrize("causal", [False, True])
def test_alibi_zero_q_closed_form(causal):
    """Q = 0 leaves only the ALiBi term: the weights of row i are
    exp(-slope |i - j|), so LSE_i = ln sum_j exp(-slope |i - j|), a sum of
    two geometric series."""
    N, H, d = 12, 2, 4
    q = torch.zeros((1, N, H, d), dtype=torch.bfloat16)
    k = rand_bf16((1, N, H, d), 41)
    v = rand_bf16((1, N, H, d), 42)
    slopes = [0.25, 1.5]
    o, lse = attn_fwd_oracle(q, k, v, 1, H, H, N, d, 1.0, causal, alibi_slopes=slopes)
    for h, a in enumerate(slopes):
        r = math.exp(-a)
        for i in range(N):
            left = (1 - r ** (i + 1)) / (1 - r)          # j = i, i-1, ..., 0
            right = 0.0 if causal else r * (1 - r ** (N - 1 - i)) / (1 - r)   # j > i
            assert abs(lse[0, h, i] - math.log(left + right)) < 1e-13
            w = np.array([r ** abs(i - j) if (j <= i or not causal) else 0.0
                          for j in range(N)])
            ref = (w[:, None] * v[0, :, h].double().numpy()).sum(0) / w.sum()
            np.testing.assert_allclose(o[0, i, h], ref, atol=1e-14, rtol=0)


def test_softcap_bounds_the_scores():
    """|cap tanh(s / cap)| < cap: each LSE lies within ln(n) +- cap, and a
    huge score range collapses to (almost) uniform weights."""
    N, H, d = 16, 2, 8
    q = rand_bf16((1, N, H, d), 51, 40.0)
    k = rand_bf16((1, N, H, d), 52, 40.0)
    v = rand_bf16((1, N, H, d), 53)
    cap = 0.05
    o, lse = attn_fwd_oracle(q, k, v, 1, H, H, N, d, 1.0, False, softcap=cap)
    assert np.all(np.abs(lse - math.log(N)) <= cap + 1e-12)
    mean_v = v[0].double().numpy().mean(0)             # [H, d]
    assert np.abs(o[0] - mean_v[None]).max() < 2 * cap * np.abs(v.double().numpy()).max()


# ---------------------------------------------------------------------------
# decode shapes: the queries are the last positions of longer key sequences
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq", [1, 3])
def test_decode_brute_force(causal, Nq):
    B, Nk, Hq, Hkv, d = 3, 13, 6, 2, 5
    kl = [13, 7, Nq]
    q = rand_bf16((B, Nq, Hq, d), 71, 2.0)
    k = rand_bf16((B, Nk, Hkv, d), 72)
    v = rand_bf16((B, Nk, Hkv, d), 73)
    o, lse = oracle.attn_decode_oracle(q, k, v, kl, causal, 0.7)
    Ob, Lb = brute_force_decode(q, k, v, kl, causal, 0.7)
    np.testing.assert_allclose(o, Ob, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, Lb, atol=1e-12, rtol=0)


def test_decode_rows_equal_the_last_prefill_rows():
    """The last Nq rows of a causal prefill over the whole sequence are the
    decode of those Nq queries against the same keys."""
    N, Nq, H, d = 40, 4, 2, 8
    q = rand_bf16((1, N, H, d), 81)
    k = rand_bf16((1, N, H, d), 82)
    v = rand_bf16((1, N, H, d), 83)
    of, lf = attn_fwd_oracle(q, k, v, 1, H, H, N, d, 0.4, True)
    od, ld = oracle.attn_decode_oracle(q[:, N - Nq:].contiguous(), k, v, [N], True, 0.4)
    np.testing.assert_array_equal(od[0], of[0, N - Nq:])
    np.testing.assert_array_equal(ld[0], lf[0, :, N - Nq:])


def test_decode_ignores_cache_rows_past_the_length():
    B, Nq, Nk, H, d = 1, 1, 20, 2, 4
    q = rand_bf16((B, Nq, H, d), 91)
    k = rand_bf16((B, Nk, H, d), 92)
    v = rand_bf16((B, Nk, H, d), 93)
    o1, l1 = oracle.attn_decode_oracle(q, k, v, [9], False, 0.5)
    k2, v2 = k.clone(), v.clone()
    k2[:, 9:] = 1e4
    v2[:, 9:] = float("nan")
    o2, l2 = oracle.attn_decode_oracle(q, k2, v2, [9], False, 0.5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ---------------------------------------------------------------------------
# paged caches: the page holding a key is read from the block table
# ---------------------------------------------------------------------------
def test_paged_decode_identity_table_is_plain_decode():
    B, Nq, Hq, Hkv, d, P, nb = 2, 2, 4, 2, 8, 4, 5
    kl = [17, 9]
    q = rand_bf16((B, Nq, Hq, d), 101)
    k = rand_bf16((B, nb * P, Hkv, d), 102)
    v = rand_bf16((B, nb * P, Hkv, d), 103)
    kc = k.reshape(B * nb, P, Hkv, d)
    vc = v.reshape(B * nb, P, Hkv, d)
    table = np.arange(B * nb).reshape(B, nb)
    for causal in (False, True):
        o1, l1 = oracle.attn_decode_paged_oracle(q, kc, vc, kl, table, P, causal, 0.5)
        o2, l2 = oracle.attn_decode_oracle(q, k, v, kl, causal, 0.5)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def test_paged_decode_is_invariant_to_page_placement():
    """Moving pages to other slots of the pool, with the table updated,
    changes nothing; pages the table does not reach are never read."""
    B, Nq, Hq, Hkv, d, P, nb = 2, 1, 4, 1, 8, 4, 4
    kl = [13, 6]
    q = rand_bf16((B, Nq, Hq, d), 111, 2.0)
    pool_k = rand_bf16((12, P, Hkv, d), 112)
    pool_v = rand_bf16((12, P, Hkv, d), 113)
    table = np.array([[3, 7, 1, 10], [0, 5, -1, -1]])
    o1, l1 = oracle.attn_decode_paged_oracle(q, pool_k, pool_v, kl, table, P, True, 0.5)
    perm = np.random.default_rng(0).permutation(12)            # new slot of old page p
    k2 = torch.empty_like(pool_k)
    v2 = torch.empty_like(pool_v)
    k2[perm] = pool_k
    v2[perm] = pool_v
    t2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1)
    for unused in set(range(12)) - set(perm[table[table >= 0]].tolist()):
        k2[unused] = float("nan")
        v2[unused] = float("nan")
    o2, l2 = oracle.attn_decode_paged_oracle(q, k2, v2, kl, t2, P, True, 0.5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ---------------------------------------------------------------------------
# backward (tang, section 3: gradients are comprehensions)
# ---------------------------------------------------------------------------
def _forward_python(q, k, v, scale, causal, g):
    """Plain Python forward of one head group: returns sum(O * G)."""
    N, H, d = len(q), len(q[0]), len(q[0][0])
    Hkv = len(k[0])
    grp = H // Hkv
    total = 0.0
    for h in range(H):
        kv = h // grp
        for i in range(N):
            js = range(i + 1) if causal else range(N)
            sc = [scale * sum(q[i][h][t] * k[j][kv][t] for t in range(d)) for j in js]
            m = max(sc)
            e = [math.exp(x - m) for x in sc]
            l = sum(e)
            for t in range(d):
                o = sum(e[n] * v[j][kv][t] for n, j in enumerate(js)) / l
                total += o * g[i][h][t]
    return total


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    """Central differences of sum(O * dO) in plain Python floats, at the
    bf16 input values, against the oracle's gradients."""
    N, Hq, Hkv, d, scale = 4, 2, 1, 3, 0.7
    q = rand_bf16((1, N, Hq, d), 121, 1.5)
    k = rand_bf16((1, N, Hkv, d), 122)
    v = rand_bf16((1, N, Hkv, d), 123)
    g = rand_bf16((1, N, Hq, d), 124)
    dq, dk, dv = oracle.attn_bwd_oracle(q, k, v, g, 1, Hq, Hkv, N, d, scale, causal)
    base = [x.float()[0].tolist() for x in (q, k, v)]
    gl = g.float()[0].tolist()
    eps = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        arr = base[which]
        for i in range(N):
            for h in range(len(arr[0])):
                for t in range(d):
                    keep = arr[i][h][t]
                    arr[i][h][t] = keep + eps
                    up = _forward_python(*base, scale, causal, gl)
                    arr[i][h][t] = keep - eps
                    dn = _forward_python(*base, scale, causal, gl)
                    arr[i][h][t] = keep
                    assert abs((up - dn) / (2 * eps) - grad[0, i, h, t]) < 1e-7


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd_fp64(causal):
    B, N, Hq, Hkv, d, scale = 2, 9, 4, 2, 6, 0.45
    q = rand_bf16((B, N, Hq, d), 131, 2.0)
    k = rand_bf16((B, N, Hkv, d), 132)
    v = rand_bf16((B, N, Hkv, d), 133)
    g = rand_bf16((B, N, Hq, d), 134)
    dq, dk, dv = oracle.attn_bwd_oracle(q, k, v, g, B, Hq, Hkv, N, d, scale, causal)
    qt, kt, vt = (x.double().requires_grad_() for x in (q, k, v))
    ke = kt.repeat_interleave(Hq // Hkv, dim=2)
    ve = vt.repeat_interleave(Hq // Hkv, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", qt, ke) * scale
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    o = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, -1), ve)
    o.backward(g.double())
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_softmax_jacobian_invariants(causal):
    """Rows of P sum to one and rows of dS to zero, so per sequence and kv
    head: sum_j dV_j = sum over the group's heads and rows of dO_i, and
    sum_j dK_j = 0."""
    lens = [7, 12]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, Hq, Hkv, d = int(cu[-1]), 6, 2, 5
    q = rand_bf16((T, Hq, d), 141, 2.0)
    k = rand_bf16((T, Hkv, d), 142)
    v = rand_bf16((T, Hkv, d), 143)
    g = rand_bf16((T, Hq, d), 144)
    dq, dk, dv = oracle.attn_bwd_oracle(q, k, v, g, 2, Hq, Hkv, T, d, 0.5, causal, cu_seqlens=cu)
    gd = g.double().numpy()
    for s in range(2):
        a, b = cu[s], cu[s + 1]
        for kv in range(Hkv):
            heads = range(kv * 3, kv * 3 + 3)
            np.testing.assert_allclose(dv[a:b, kv].sum(0), gd[a:b, list(heads)].sum((0, 1)),
                                       atol=1e-12, rtol=0)
            np.testing.assert_allclose(dk[a:b, kv].sum(0), 0.0, atol=1e-12)
