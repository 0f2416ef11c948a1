"""Pins for the fp64 CPU oracle, against things other than the oracle itself:
closed forms, a high-precision brute force written independently (mpmath,
log-sum-exp without the max shift), permutation structure, block-size
invariance of the online softmax, finite differences, and the E4M3 format
checked against torch's cast.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- brute force
def need_mpmath():
    """The high-precision brute force needs mpmath; only the tests that use it are
    skipped without it (every other pin in this file runs regardless)."""
    return pytest.importorskip("mpmath")


def mp_forward(q, k, v, scale, causal, dps=40):
    """Independent high-precision brute force: lse_i = log sum_j exp(S_ij) with
    no max shift, O_i = sum_j exp(S_ij - lse_i) V_j."""
    mpmath = need_mpmath()
    with mpmath.workdps(dps):
        N, d = q.shape
        O = [[mpmath.mpf(0)] * d for _ in range(N)]
        lse = []
        for i in range(N):
            keys = [j for j in range(N) if not (causal and j > i)]
            s = {j: mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[i, c]) * mpmath.mpf(k[j, c])
                                                   for c in range(d)) for j in keys}
            L = mpmath.log(mpmath.fsum(mpmath.exp(s[j]) for j in keys))
            lse.append(L)
            for c in range(d):
                O[i][c] = mpmath.fsum(mpmath.exp(s[j] - L) * mpmath.mpf(v[j, c]) for j in keys)
        return O, lse


def to_np(O):
    return np.array([[float(x) for x in row] for row in O])


@pytest.mark.parametrize("N,d,causal,scale", [(1, 3, False, 0.7), (4, 3, False, 0.5),
                                              (5, 2, True, 1.3), (6, 4, False, 2.0),
                                              (6, 4, True, 0.25)])
def test_fwd_matches_brute_force(N, d, causal, scale):
    q, k, v = rnd(1, N, d), rnd(2, N, d), rnd(3, N, d)
    o, lse = oracle.attn_fwd(q, k, v, scale, causal)
    O_mp, lse_mp = mp_forward(q, k, v, scale, causal)
    np.testing.assert_allclose(o, to_np(O_mp), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, [float(x) for x in lse_mp], rtol=0, atol=1e-13)


def test_fwd_large_scores_stay_finite():
    # scores ~ +-1e3: exp would overflow without the max shift
    N, d = 5, 3
    q, k, v = 30 * rnd(4, N, d), 30 * rnd(5, N, d), rnd(6, N, d)
    o, lse = oracle.attn_fwd(q, k, v, 1.0, False)
    O_mp, lse_mp = mp_forward(q, k, v, 1.0, False, dps=60)
    assert np.all(np.isfinite(o))
    np.testing.assert_allclose(o, to_np(O_mp), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, [float(x) for x in lse_mp], rtol=1e-14)


# ---------------------------------------------------------------- closed forms
def test_two_by_two_worked_example():
    # Q = K = I, V = [[1,2],[3,4]], scale 1: S = I, row softmax of (1,0) and (0,1)
    q = np.eye(2)
    v = np.array([[1.0, 2.0], [3.0, 4.0]])
    o, lse = oracle.attn_fwd(q, q, v, 1.0)
    e = math.e
    np.testing.assert_allclose(o[0], (e * v[0] + v[1]) / (e + 1), atol=1e-15)
    np.testing.assert_allclose(o[1], (v[0] + e * v[1]) / (e + 1), atol=1e-15)
    np.testing.assert_allclose(lse, [math.log(e + 1)] * 2, atol=1e-15)
    # causal: row 0 sees key 0 only; row 1 is unchanged
    oc, lsec = oracle.attn_fwd(q, q, v, 1.0, causal=True)
    np.testing.assert_allclose(oc[0], v[0], atol=1e-15)
    np.testing.assert_allclose(oc[1], o[1], atol=1e-15)
    np.testing.assert_allclose(lsec[0], 1.0, atol=1e-15)


def test_single_key_returns_v():
    q, k, v = rnd(7, 3, 1, 5), rnd(8, 3, 1, 5), rnd(9, 3, 1, 5)
    o, lse = oracle.attn_fwd(q, k, v, 0.3)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.3 * np.sum(q * k, axis=-1), atol=1e-14)


def test_zero_scale_is_mean_of_v():
    N, d = 9, 4
    q, k, v = rnd(10, N, d), rnd(11, N, d), rnd(12, N, d)
    o, lse = oracle.attn_fwd(q, k, v, 0.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), (N, d)), atol=1e-14)
    np.testing.assert_allclose(lse, np.log(N), atol=1e-14)
    oc, lsec = oracle.attn_fwd(q, k, v, 0.0, causal=True)
    prefix_mean = np.cumsum(v, 0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(oc, prefix_mean, atol=1e-14)
    np.testing.assert_allclose(lsec, np.log(np.arange(1, N + 1)), atol=1e-14)


def test_constant_v_gives_constant_o():
    N, d = 11, 3
    q, k = rnd(13, N, d), rnd(14, N, d)
    v = np.full((N, d), 2.5)
    for causal in (False, True):
        o, _ = oracle.attn_fwd(q, k, v, 0.9, causal)
        np.testing.assert_allclose(o, 2.5, atol=1e-14)


def test_causal_first_row_is_v0():
    q, k, v = rnd(15, 2, 7, 4), rnd(16, 2, 7, 4), rnd(17, 2, 7, 4)
    o, _ = oracle.attn_fwd(q, k, v, 1.0, causal=True)
    np.testing.assert_allclose(o[:, 0], v[:, 0], atol=1e-15)


def test_one_hot_dominant_score():
    # row 2's query points along a direction u; scaled so the best key beats the
    # runner-up by > 40 nats, O_2 is that key's value to ~exp(-40)
    N, d = 8, 4
    k = rnd(18, N, d)
    v = rnd(19, N, d)
    u = rnd(65, d)
    proj = k @ u
    best = int(np.argmax(proj))
    gap = proj[best] - np.sort(proj)[-2]
    q = np.zeros((N, d))
    q[2] = (45.0 / gap) * u
    o, _ = oracle.attn_fwd(q, k, v, 1.0)
    np.testing.assert_allclose(o[2], v[best], atol=1e-12)
    # rows with q = 0 see uniform weights
    np.testing.assert_allclose(o[0], v.mean(0), atol=1e-14)


def test_softmax_rows_sum_to_one():
    # with V = I (N x N), O is P itself
    N = 13
    q, k = rnd(20, N, N), rnd(21, N, N)
    for causal in (False, True):
        P, _ = oracle.attn_fwd(q, k, np.eye(N), 0.4, causal)
        np.testing.assert_allclose(P.sum(1), 1.0, atol=1e-14)
        assert np.all(P >= 0)
        if causal:
            assert np.all(np.triu(P, 1) == 0)


def test_shift_invariance_of_scores():
    # adding c_i to every score of row i leaves P unchanged and shifts lse by c_i:
    # append feature c_i to q_i and a constant 1 to every k_j (v padded with 0)
    N, d = 10, 3
    q, k, v = rnd(22, N, d), rnd(23, N, d), rnd(24, N, d)
    o1, lse1 = oracle.attn_fwd(q, k, v, 1.0)
    shift = rnd(25, N)
    q2 = np.concatenate([q, shift[:, None]], 1)
    k2 = np.concatenate([k, np.ones((N, 1))], 1)
    vpad = np.concatenate([v, np.zeros((N, 1))], 1)
    o2, lse2 = oracle.attn_fwd(q2, k2, vpad, 1.0)
    np.testing.assert_allclose(o2[:, :d], o1, atol=1e-13)
    np.testing.assert_allclose(lse2, lse1 + shift, atol=1e-13)


# ---------------------------------------------------------------- structure
def test_permutation_equivariance():
    N, d = 12, 5
    q, k, v = rnd(26, N, d), rnd(27, N, d), rnd(28, N, d)
    o, lse = oracle.attn_fwd(q, k, v, 0.8)
    perm = np.random.default_rng(29).permutation(N)
    oq, lseq = oracle.attn_fwd(q[perm], k, v, 0.8)
    np.testing.assert_allclose(oq, o[perm], atol=1e-14)
    np.testing.assert_allclose(lseq, lse[perm], atol=1e-14)
    okv, lsekv = oracle.attn_fwd(q, k[perm], v[perm], 0.8)
    np.testing.assert_allclose(okv, o, atol=1e-14)
    np.testing.assert_allclose(lsekv, lse, atol=1e-14)


def test_heads_are_independent():
    q, k, v = rnd(30, 2, 3, 6, 4), rnd(31, 2, 3, 6, 4), rnd(32, 2, 3, 6, 4)
    o, lse = oracle.attn_fwd(q, k, v, 0.5, True)
    for b in range(2):
        for h in range(3):
            ob, lb = oracle.attn_fwd(q[b, h], k[b, h], v[b, h], 0.5, True)
            np.testing.assert_array_equal(o[b, h], ob)
            np.testing.assert_array_equal(lse[b, h], lb)


def test_rows_entry_matches_full():
    N, d = 40, 8
    q, k, v = rnd(33, N, d), rnd(34, N, d), rnd(35, N, d)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, 0.35, causal)
        rows = [0, 3, 17, 39, 3]
        orr, lser = oracle.attn_fwd_rows(q, k, v, rows, 0.35, causal)
        np.testing.assert_array_equal(orr, o[rows])
        np.testing.assert_array_equal(lser, lse[rows])


# ---------------------------------------------------------------- online softmax
@pytest.mark.parametrize("N", [1, 37, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_is_block_size_independent(N, causal):
    d = 8
    q, k, v = rnd(36, 2, N, d), rnd(37, 2, N, d), rnd(38, 2, N, d)
    ref, lse_ref = oracle.attn_fwd(q, k, v, 1 / math.sqrt(d), causal)
    for Br, Bc in [(1, 1), (7, 7), (32, 32), (128, 128), (N, N), (7, 32), (32, 7), (N, 1)]:
        o, lse = oracle.attn_fwd_tiled(q, k, v, Br, Bc, 1 / math.sqrt(d), causal)
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)


def test_p1_numpy_demo_configuration():
    cfg = json.load(open(os.path.join(GOLDEN, "p1_numpy_demo.json")))
    rs = np.random.RandomState(cfg["seed"])
    n, d = cfg["n"], cfg["d"]
    Q, K, V = rs.randn(n, d), rs.randn(n, d), rs.randn(n, d)
    tiled, _ = oracle.attn_fwd_tiled(Q, K, V, cfg["block_size"], cfg["block_size"],
                                     1 / math.sqrt(d))
    ref, _ = oracle.attn_fwd(Q, K, V, 1 / math.sqrt(d))
    err = np.abs(tiled - ref).max()
    assert err < cfg["max_abs_err_bar"]
    assert err < 1e-13  # fp64 throughout: rounding level


def test_p3_fp32_scale_plausibility():
    # The page's float32 block simulation differs from standard attention by
    # ~3e-7 at N=128, d=64, Br=Bc=32; float32 rounding of the fp64 oracle's
    # output lands on the same scale.
    cfg = json.load(open(os.path.join(GOLDEN, "p3_fp32_errors.json")))
    N, d = cfg["N"], cfg["d"]
    q, k, v = rnd(39, N, d), rnd(40, N, d), rnd(41, N, d)
    o, _ = oracle.attn_fwd(q, k, v, 1 / math.sqrt(d))
    t, _ = oracle.attn_fwd_tiled(q.astype(np.float32), k.astype(np.float32),
                                 v.astype(np.float32), cfg["Br"], cfg["Bc"], 1 / math.sqrt(d))
    rounding = np.abs(o.astype(np.float32).astype(np.float64) - o).max()
    assert rounding < 10 * cfg["fwd_max_abs_err"]
    # inputs rounded to fp32 move the result by far less than the 1e-5 fp32 bar
    assert np.abs(t - o).max() < 1e-5


# ---------------------------------------------------------------- backward
def mp_grad_fd(q, k, v, do, scale, causal, h=1e-12, dps=50):
    """Central finite differences of L = <dO, O> through the mpmath forward."""
    mpmath = need_mpmath()
    grads = []
    for which in range(3):
        base = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(q)
        for idx in np.ndindex(*q.shape):
            vals = []
            for sgn in (+1, -1):
                with mpmath.workdps(dps):
                    xs = [np.vectorize(mpmath.mpf, otypes=[object])(x) for x in base]
                    xs[which][idx] = xs[which][idx] + sgn * mpmath.mpf(h)
                    O, _ = mp_forward_obj(xs[0], xs[1], xs[2], scale, causal, dps)
                    vals.append(mpmath.fsum(O[i][c] * mpmath.mpf(do[i, c])
                                            for i in range(q.shape[0])
                                            for c in range(q.shape[1])))
            with mpmath.workdps(dps):
                g[idx] = float((vals[0] - vals[1]) / (2 * mpmath.mpf(h)))
        grads.append(g)
    return grads


def mp_forward_obj(q, k, v, scale, causal, dps):
    mpmath = need_mpmath()
    with mpmath.workdps(dps):
        N, d = q.shape
        O = [[None] * d for _ in range(N)]
        for i in range(N):
            keys = [j for j in range(N) if not (causal and j > i)]
            s = {j: mpmath.mpf(scale) * mpmath.fsum(q[i, c] * k[j, c] for c in range(d))
                 for j in keys}
            L = mpmath.log(mpmath.fsum(mpmath.exp(s[j]) for j in keys))
            for c in range(d):
                O[i][c] = mpmath.fsum(mpmath.exp(s[j] - L) * v[j, c] for j in keys)
        return O, None


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_matches_finite_differences(causal):
    N, d, scale = 4, 3, 0.7
    q, k, v, do = rnd(42, N, d), rnd(43, N, d), rnd(44, N, d), rnd(45, N, d)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale, causal)
    fq, fk, fv = mp_grad_fd(q, k, v, do, scale, causal)
    for got, want in ((dq, fq), (dk, fk), (dv, fv)):
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_bwd_fd_fp64_larger():
    # fp64 central differences through the oracle's forward at a larger shape
    N, d, scale, h = 7, 4, 0.9, 1e-6
    q, k, v, do = rnd(46, N, d), rnd(47, N, d), rnd(48, N, d), rnd(49, N, d)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale, False)

    def L(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, scale)
        return float(np.sum(o * do))

    for which, got in enumerate((dq, dk, dv)):
        for idx in [(0, 0), (3, 2), (6, 3), (5, 1)]:
            xs_p = [q.copy(), k.copy(), v.copy()]
            xs_m = [q.copy(), k.copy(), v.copy()]
            xs_p[which][idx] += h
            xs_m[which][idx] -= h
            fd = (L(*xs_p) - L(*xs_m)) / (2 * h)
            assert abs(fd - got[idx]) <= 1e-7 * max(1.0, abs(fd))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_sum_identities(causal):
    N, d = 33, 6
    q, k, v, do = rnd(50, N, d), rnd(51, N, d), rnd(52, N, d), rnd(53, N, d)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.5, causal)
    # rows of P sum to 1  =>  sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(0), do.sum(0), atol=1e-12)
    # rows of dS sum to delta_i - delta_i = 0  =>  sum_j dK_j = 0
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-12)


def test_bwd_single_key():
    # N = 1: O = V regardless of Q, K  =>  dQ = dK = 0, dV = dO
    q, k, v, do = rnd(54, 1, 4), rnd(55, 1, 4), rnd(56, 1, 4), rnd(57, 1, 4)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 1.0)
    np.testing.assert_allclose(dq, 0, atol=1e-15)
    np.testing.assert_allclose(dk, 0, atol=1e-15)
    np.testing.assert_allclose(dv, do, atol=1e-15)


def test_bwd_is_linear_in_dout():
    N, d = 9, 3
    q, k, v = rnd(58, N, d), rnd(59, N, d), rnd(60, N, d)
    a, b = rnd(61, N, d), rnd(62, N, d)
    ga = oracle.attn_bwd(q, k, v, a, 0.6)
    gb = oracle.attn_bwd(q, k, v, b, 0.6)
    gab = oracle.attn_bwd(q, k, v, 2 * a - 3 * b, 0.6)
    for x, y, z in zip(ga, gb, gab):
        np.testing.assert_allclose(z, 2 * x - 3 * y, atol=1e-12)


# ---------------------------------------------------------------- E4M3
def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    np.testing.assert_array_equal(mine[~nan], ref[~nan])


def test_e4m3_format_landmarks():
    d = oracle.e4m3_decode
    assert d([0x7E])[0] == 448.0                       # largest finite
    assert d([0x01])[0] == 2.0 ** -9                   # smallest subnormal
    assert d([0x08])[0] == 2.0 ** -6                   # smallest normal
    assert d([0x38])[0] == 1.0
    assert d([0xB8])[0] == -1.0
    assert d([0x3A], 0.5)[0] == 1.25 * 0.5             # descale multiplies


def test_e4m3_encode_matches_torch_rne():
    x = np.concatenate([np.random.default_rng(63).standard_normal(20000) * 50,
                        np.random.default_rng(64).standard_normal(2000) * 0.01,
                        [0.0, -0.0, 448.0, 447.9, -449.0, 1e6, 2.0 ** -10, 3 * 2.0 ** -10]])
    mine = oracle.e4m3_encode(x)
    clamped = np.clip(x, -448, 448)
    ref = torch.from_numpy(clamped).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(mine, ref)
    # every finite code round-trips
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_bwd_matches_finite_differences_of_shared_kv(causal):
    # grouped-query: 4 query heads share 2 K/V heads.  Perturbing one element of a
    # shared K or V head moves every query head of its group, so the finite
    # difference of L = <dO, O> checks the group sum (a gradient taken from one
    # query head only, or summed over the wrong group, fails here).
    B, H, H_kv, N, d, scale, h = 1, 4, 2, 5, 3, 0.8, 1e-6
    q, do = rnd(60, B, H, N, d), rnd(61, B, H, N, d)
    k, v = rnd(62, B, H_kv, N, d), rnd(63, B, H_kv, N, d)
    dq, dk, dv = oracle.attn_bwd_gqa(q, k, v, do, scale, causal)
    assert dk.shape == k.shape and dv.shape == v.shape and dq.shape == q.shape

    def L(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, np.repeat(kk, 2, axis=1), np.repeat(vv, 2, axis=1), scale,
                               causal)
        return float(np.sum(o * do))

    for which, got in enumerate((dq, dk, dv)):
        for idx in [(0, 0, 0, 0), (0, 1, 4, 2), (0, 1, 2, 1)] + ([(0, 3, 3, 0)] if which == 0 else []):
            xs_p = [q.copy(), k.copy(), v.copy()]
            xs_m = [q.copy(), k.copy(), v.copy()]
            xs_p[which][idx] += h
            xs_m[which][idx] -= h
            fd = (L(*xs_p) - L(*xs_m)) / (2 * h)
            assert abs(fd - got[idx]) <= 1e-7 * max(1.0, abs(fd))


def test_gqa_with_one_group_per_head_is_plain_attention():
    # H_kv = H: the grouped entry points reduce to the plain ones
    q, k, v, do = (rnd(70 + i, 2, 3, 6, 4) for i in range(4))
    a = oracle.attn_bwd_gqa(q, k, v, do, 0.5, True)
    b = oracle.attn_bwd(q, k, v, do, 0.5, True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    with pytest.raises(ValueError):
        oracle.attn_fwd_gqa(q, k[:, :2], v[:, :2], 0.5)


# ---- key shards and the lse merge ("FlashAttention-1" 10.2.2 combination rule)

@pytest.mark.parametrize("causal", [False, True])
def test_kv_shard_whole_sequence_is_the_forward(causal):
    # one shard holding every key is plain attention: the numpy shard oracle
    # against the C oracle (two independent codings of 10.2.1)
    q, k, v = rnd(80, 2, 9, 5), rnd(81, 2, 9, 5), rnd(82, 2, 9, 5)
    o1, l1 = oracle.attn_fwd_kv_shard(q, k, v, 0.7, causal)
    o2, l2 = oracle.attn_fwd(q, k, v, 0.7, causal)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("cuts", [(4,), (1, 7), (3, 5, 6), (0, 2, 11)])
def test_merging_key_shards_gives_the_full_forward(causal, cuts):
    # split the keys at `cuts`, attend each shard with its global offset, merge:
    # the full forward of the C oracle.  A wrong merge weight, a dropped shard or a
    # causal offset of the wrong sign fails here.
    N, d = 12, 4
    q, k, v = rnd(83, 1, 2, N, d), rnd(84, 1, 2, N, d), rnd(85, 1, 2, N, d)
    edges = [0, *cuts, N]
    parts = [oracle.attn_fwd_kv_shard(q, k[..., a:b, :], v[..., a:b, :], 0.9, causal,
                                      q_offset=0, kv_offset=a)
             for a, b in zip(edges[:-1], edges[1:])]
    o, lse = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, 0.9, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)


def test_query_shards_with_offsets_tile_the_causal_forward():
    # queries split as well: block (qa..qb) x (ka..kb) with both offsets, merged
    # over the key shards, equals the rows qa..qb of the full causal forward
    N, d = 10, 3
    q, k, v = rnd(86, N, d), rnd(87, N, d), rnd(88, N, d)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, 1.1, True)
    edges = [0, 3, 8, 10]
    for qa, qb in zip(edges[:-1], edges[1:]):
        parts = [oracle.attn_fwd_kv_shard(q[qa:qb], k[ka:kb], v[ka:kb], 1.1, True, qa, ka)
                 for ka, kb in zip(edges[:-1], edges[1:])]
        o, lse = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        np.testing.assert_allclose(o, o_ref[qa:qb], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref[qa:qb], rtol=0, atol=1e-13)


def test_kv_shard_rows_that_see_no_key():
    # keys 5.. against queries 0..3 under the causal mask: nothing visible
    q, k, v = rnd(89, 4, 3), rnd(90, 2, 3), rnd(91, 2, 3)
    o, lse = oracle.attn_fwd_kv_shard(q, k, v, 1.0, True, q_offset=0, kv_offset=5)
    assert np.all(o == 0) and np.all(lse == -np.inf)
    # query 5 sees exactly key 5: O = V_0 of the shard, lse = scale q.k
    o, lse = oracle.attn_fwd_kv_shard(q, k, v, 1.0, True, q_offset=2, kv_offset=5)
    assert np.all(o[:3] == 0) and np.all(lse[:3] == -np.inf)
    np.testing.assert_allclose(o[3], v[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[3], q[3] @ k[0], rtol=0, atol=1e-14)


def test_lse_merge_closed_forms():
    o_a, o_b = rnd(92, 5, 4), rnd(93, 5, 4)
    # two parts of equal weight: the mean, and lse + ln 2
    o, lse = oracle.lse_merge(np.stack([o_a, o_b]), np.full((2, 5), 1.5))
    np.testing.assert_allclose(o, (o_a + o_b) / 2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 1.5 + math.log(2), rtol=0, atol=1e-15)
    # weights e^1 : e^3 -> O = (o_a + e^2 o_b) / (1 + e^2), lse = ln(e + e^3)
    o, lse = oracle.lse_merge(np.stack([o_a, o_b]), np.stack([np.full(5, 1.0), np.full(5, 3.0)]))
    w = math.exp(2.0)
    np.testing.assert_allclose(o, (o_a + w * o_b) / (1 + w), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(math.e + math.e ** 3), rtol=0, atol=1e-14)
    # a -inf part drops out whatever its O holds; all -inf gives O = 0, lse = -inf
    lse_in = np.stack([np.full(5, -np.inf), np.full(5, 0.25)])
    o, lse = oracle.lse_merge(np.stack([o_a, o_b]), lse_in)
    np.testing.assert_array_equal(o, o_b)
    np.testing.assert_array_equal(lse, np.full(5, 0.25))
    o, lse = oracle.lse_merge(np.stack([o_a, o_b]), np.full((2, 5), -np.inf))
    assert np.all(o == 0) and np.all(lse == -np.inf)
    # very different magnitudes stay finite (the merge subtracts the max)
    o, lse = oracle.lse_merge(np.stack([o_a, o_b]), np.stack([np.full(5, 800.0), np.full(5, -800.0)]))
    np.testing.assert_allclose(o, o_a, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 800.0, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- per-block E4M3 factors
def test_e4m3_decode_blocks_constant_factor_is_per_tensor_decode():
    # one factor for every block is the per-tensor dequantisation
    codes = np.random.default_rng(7).integers(0, 256, size=(2, 3, 300, 8), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0  # drop the NaN codes
    got = oracle.e4m3_decode_blocks(codes, np.full((2, 3, 3), 0.375))
    np.testing.assert_array_equal(got, oracle.e4m3_decode(codes, 0.375))


def test_e4m3_decode_blocks_factor_reaches_exactly_its_rows():
    # Doubling an E4M3 value of magnitude <= 224 is exact.  Doubling the codes of rows
    # 128..255 and halving block 1's factor must give identical values, and doubling
    # the factor of block 2 (rows 256..299, a short block) must double only those rows.
    rng = np.random.default_rng(8)
    vals = rng.uniform(-200.0, 200.0, size=(300, 16))
    codes = oracle.e4m3_encode(vals)
    f = np.array([0.5, 0.25, 2.0])
    base = oracle.e4m3_decode_blocks(codes, f)
    codes2 = codes.copy()
    codes2[128:256] = oracle.e4m3_encode(2.0 * oracle.e4m3_decode(codes[128:256]))
    f2 = f.copy()
    f2[1] /= 2
    np.testing.assert_array_equal(oracle.e4m3_decode_blocks(codes2, f2), base)
    f3 = f.copy()
    f3[2] *= 2
    got = oracle.e4m3_decode_blocks(codes, f3)
    np.testing.assert_array_equal(got[:256], base[:256])
    np.testing.assert_array_equal(got[256:], 2.0 * base[256:])
    # row i has factor f[i // 128]
    dec = oracle.e4m3_decode(codes)
    for i in (0, 127, 128, 255, 256, 299):
        np.testing.assert_array_equal(base[i], dec[i] * f[i // 128])


def test_e4m3_decode_blocks_rejects_wrong_block_count():
    codes = np.zeros((300, 4), dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle.e4m3_decode_blocks(codes, np.ones(2))
