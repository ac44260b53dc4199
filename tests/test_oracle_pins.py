"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each checks a closed form, an
exact (rational / integer) computation, a textbook special case, a hand-worked
fixture under tests/golden/, or an invariant of the method.  Sources: Quant
VideoGen explainer (Sommario tecnico sec. 2A SAS, sec. 2B PRQ, sec. 3 centroid
caching, sec. 4 "up to 7x", baselines RTN/KIVI), Coral-KV news items
("cross-layer prediction": block-diagonal per head plus global low rank), and
for the attention that consumes the cache the explainer's sec. 3 (fused
dequantisation) with the 33-method Self-Forcing KV-cache study's abstract.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from synth import synth as SY
from synth import workloads as WL

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------- helpers ---

def bf16_fraction(b):
    """Exact rational value of a bf16 bit pattern."""
    b = int(b)
    sign = -1 if b & 0x8000 else 1
    e = (b >> 7) & 0xFF
    m = b & 0x7F
    if e == 0:
        return sign * Fraction(m, 1 << 133)
    return sign * Fraction(128 + m, 1) * Fraction(2) ** (e - 134)


def round_fraction_to_bf16(v):
    """Correct round-to-nearest-even of an exact rational to bf16 bits
    (normal range)."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    # a in [1, 2): significand with 7 fraction bits
    n = a * 128
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    if fl == 256:
        fl = 128
        e += 1
    return sign | ((e + 127) << 7) | (fl - 128)


def rand_bf16(rng, shape, scale=1.0):
    return SY.f64_to_bf16_bits(rng.standard_normal(shape) * scale)


def f32(b):
    return SY.bf16_bits_to_f32(b)


def decode_meta(meta):
    s = (meta & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float32)
    z = (meta >> 16).astype(np.uint16).view(np.float16).astype(np.float32)
    return s, z


def unpack(codes, D, b=2):
    """codes [..., D*b/32] uint32 -> [..., D] ints (b-bit fields, least
    significant first)."""
    per = 32 // b
    sh = (b * np.arange(per, dtype=np.uint32))
    q = (codes[..., :, None] >> sh) & np.uint32((1 << b) - 1)
    return q.reshape(codes.shape[:-1] + (D,)).astype(np.int64)


# --------------------------------------------------------------- formats ---

def test_bf16_rounding_is_exact_nearest_even(oracle):
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(400) * 10.0 ** rng.integers(-6, 6, 400))
    # exact midpoints between neighbouring bf16 values (ties to even)
    for b in (0x3F80, 0x3F81, 0x4000, 0xC123, 0x0080):
        lo, hi = bf16_fraction(b), bf16_fraction(b + 1)
        vals.append(float((lo + hi) / 2))
    for v in vals:
        assert oracle.to_bf16(v) == round_fraction_to_bf16(Fraction(v)), v


def test_f16_rounding_matches_ieee(oracle):
    rng = np.random.default_rng(2)
    v = np.concatenate([
        (rng.standard_normal(2000) * 10.0 ** rng.integers(-9, 5, 2000)).astype(np.float32),
        np.float32([65504, 65519.99, 65520, 6.1e-5, 5.96e-8, 2.98e-8, 1e-9, 0.0, -0.0, 2049, 2051]),
    ])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)   # IEEE round-to-nearest-even
    got = np.array([oracle.to_f16(x) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)
    back = np.array([oracle.f16_to_f32(h) for h in ref], dtype=np.float32)
    assert np.array_equal(back, ref.view(np.float16).astype(np.float32))


# ------------------------------------------------- PRQ / group quantiser ---

def rtn_reference(xb, G, b=2):
    """Plain b-bit asymmetric group round-to-nearest (the RTN baseline), one
    stage, no smoothing; vectorised numpy fp32: q = clip(rint((x - z) / s)),
    numpy's float32 division being IEEE division."""
    L = (1 << b) - 1
    x = f32(xb)
    N, D = x.shape
    g = x.reshape(N, D // G, G)
    mn, mx = g.min(-1), g.max(-1)
    s16 = ((mx - mn) / np.float32(L)).astype(np.float16)
    z16 = mn.astype(np.float16)
    s, z = s16.astype(np.float32), z16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(s[..., None] != 0, (g - z[..., None]) / s[..., None], np.float32(0)).astype(np.float32)
    q = np.clip(np.rint(t), 0, L).astype(np.uint32)
    per = 32 // b
    q = q.reshape(N, D // per, per)
    codes = (q << (b * np.arange(per, dtype=np.uint32))).sum(-1, dtype=np.uint64).astype(np.uint32)
    meta = s16.view(np.uint16).astype(np.uint32) | (z16.view(np.uint16).astype(np.uint32) << 16)
    return codes, meta


@pytest.mark.parametrize("D,G,b", [(64, 64, 2), (128, 64, 2), (128, 128, 2), (128, 32, 2),
                                   (64, 64, 4), (128, 64, 4), (128, 16, 4)])
def test_single_stage_no_smoothing_is_rtn(oracle, D, G, b):
    rng = np.random.default_rng(D + G + b)
    x = rand_bf16(rng, (300, D), 2.0)
    codes, meta = oracle.prq_encode(x, None, None, 1, G, b)
    rc, rm = rtn_reference(x, G, b)
    assert np.array_equal(codes[0], rc)
    assert np.array_equal(meta[0], rm)


def _midpoint_scales(bits, L, kmax):
    """Every fp16 scale s = m * 2^e with a `bits`-bit significand m, over 20
    binades, for which 0, L*s and the midpoints (k + 1/2)*s, k <= kmax, are all
    exact in bf16."""
    out = []
    for e in range(-14, 6):
        for m in range(1 << (bits - 1), 1 << bits):
            s = m * 2.0 ** (e - bits + 1)
            vals = np.array([0.0, L * s] + [(k + 0.5) * s for k in range(kmax + 1)])
            if float(np.float16(s)) == s and np.array_equal(
                    f32(SY.f64_to_bf16_bits(vals)).astype(np.float64), vals):
                out.append(s)
    return out


@pytest.mark.parametrize("b", [2, 4])
def test_exact_midpoints_round_to_even_level(oracle, b):
    """An element exactly halfway between levels k and k+1 ((r - z)/s = k + 1/2
    as an exact quotient) is coded to the even one of the two, for every scale
    of a given width -- the rint-to-even rule applied to the exact quotient.
    Groups are [0, L*s, midpoints...]: min 0 gives z = 0, and L*s / L = s
    exactly.  A quantiser that rounds (r - z) * fp32(1/s) instead misses some of
    these (at about one scale in five the product lands one float below or
    above the midpoint)."""
    L = (1 << b) - 1
    kmax = 2 if b == 2 else 7          # midpoints (k + 1/2) s still exact in bf16
    scales = _midpoint_scales(6 if b == 2 else 5, L, kmax)
    assert len(scales) >= 150
    D = G = 64
    mids = [(k + 0.5) for k in range(kmax + 1)]
    rows, want = [], []
    for s in scales:
        vals = [0.0, L * s] + [m * s for m in mids]
        codes = [0, L] + [int(k + 1) if (k + 1) % 2 == 0 else int(k) for k in range(kmax + 1)]
        reps = D // len(vals) + 1
        rows.append((vals * reps)[:D])
        want.append((codes * reps)[:D])
    x = SY.f64_to_bf16_bits(np.array(rows))
    assert np.array_equal(f32(x).astype(np.float64), np.array(rows))      # the values are exact
    got_codes, meta = oracle.prq_encode(x, None, None, 1, G, b)
    s_got, z_got = decode_meta(meta[0][:, 0])
    assert np.array_equal(s_got.astype(np.float64), np.array(scales)) and np.all(z_got == 0)
    assert np.array_equal(unpack(got_codes[0], D, b), np.array(want))


def test_pack_example_golden(oracle):
    fx = {}
    for line in open(os.path.join(GOLD, "pack_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        fx[k] = v
    pat = [int(h, 16) for h in fx["row_bf16"]]
    row = np.array([pat[j % 4] for j in range(64)], np.uint16)[None, :]
    codes, meta = oracle.prq_encode(row, None, None, 1, 64)
    assert codes.shape == (1, 1, int(fx["words_per_row"][0]))
    assert all(int(w) == int(fx["codes_word"][0], 16) for w in codes[0, 0])
    assert int(meta[0, 0, 0]) == int(fx["meta_word"][0], 16)
    out = oracle.decode(codes, meta, None, None, 64)
    assert np.array_equal(out, row)


def test_pack_example_4bit_golden(oracle):
    """The hand-worked 4-bit row of tests/golden/pack_example_4bit.txt."""
    fx = {}
    for line in open(os.path.join(GOLD, "pack_example_4bit.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        fx[k] = v
    pat = [int(h, 16) for h in fx["row_bf16"]]
    row = np.array([pat[j % 16] for j in range(64)], np.uint16)[None, :]
    codes, meta = oracle.prq_encode(row, None, None, 1, 64, 4)
    assert codes.shape == (1, 1, int(fx["words_per_row"][0]))
    want = [int(w, 16) for w in fx["codes_words"]]
    assert [int(w) for w in codes[0, 0]] == want * 4
    assert int(meta[0, 0, 0]) == int(fx["meta_word"][0], 16)
    assert np.array_equal(oracle.decode(codes, meta, None, None, 64, 4), row)


@pytest.mark.parametrize("b", [2, 4])
def test_on_grid_values_round_trip(oracle, b):
    """Groups whose values are exactly z + k*s (s, z fp16, k in 0..L with
    L = 2^b - 1, every level present) decode exactly and give codes k."""
    rng = np.random.default_rng(3 if b == 2 else 7)
    D, G, L = 128, 64, (1 << b) - 1
    rows, ks = [], []
    for _ in range(50):
        row, krow = [], []
        for g in range(D // G):
            s = float(np.float16(2.0 ** rng.integers(-6, 2)))
            # b = 4: z a multiple of s, so that every z + k*s = (m + k)*s,
            # |m + k| < 256, is exact in bf16
            z = float(np.float16(rng.integers(-64, 64) * (2.0 ** -4 if b == 2 else s)))
            k = rng.integers(0, L + 1, G)
            k[:L + 1] = np.arange(L + 1)
            rng.shuffle(k)
            row += [z + kk * s for kk in k]
            krow += list(k)
        rows.append(row)
        ks.append(krow)
    x = SY.f64_to_bf16_bits(np.array(rows))
    assert np.array_equal(f32(x).astype(np.float64), np.array(rows))   # exact in bf16
    codes, meta = oracle.prq_encode(x, None, None, 1, G, b)
    assert np.array_equal(unpack(codes[0], D, b), np.array(ks))
    assert np.array_equal(oracle.decode(codes, meta, None, None, G, b), x)


@pytest.mark.parametrize("b", [2, 4])
def test_constant_group(oracle, b):
    x = np.full((4, 64), 0x3FC0, np.uint16)    # 1.5 everywhere
    codes, meta = oracle.prq_encode(x, None, None, 2, 64, b)
    assert codes.shape == (2, 4, 64 * b // 32)
    s, z = decode_meta(meta)
    assert np.all(s == 0) and np.all(z[0] == 1.5) and np.all(z[1] == 0)
    assert np.all(codes == 0)
    assert np.array_equal(oracle.decode(codes, meta, None, None, 64, b), x)


def per_stage_residuals(x, S, G, oracle, b=2):
    """Residual after each number of stages, rebuilt from the stored codes
    (fp64 arithmetic of the dequantised values)."""
    codes, meta = oracle.prq_encode(x, None, None, S, G, b)
    N, D = x.shape
    s, z = decode_meta(meta)
    q = unpack(codes, D, b).astype(np.float64)
    rng_s = np.repeat(s.astype(np.float64), G, axis=-1)
    rng_z = np.repeat(z.astype(np.float64), G, axis=-1)
    deq = q * rng_s + rng_z
    r = f32(x).astype(np.float64)
    out = [r.copy()]
    for k in range(S):
        r = r - deq[k]
        out.append(r.copy())
    return out, s, z


@pytest.mark.parametrize("b", [2, 4])
def test_stage_error_bound_and_monotonicity(oracle, b):
    """|r_s - deq_s| <= s/2 + fp16 slack per element, and the per-group max-abs
    error after a stage is at most (max-min of its input)/(2L) + slack with
    L = 2^b - 1, so it does not grow as stages are added (PRQ items 1-2)."""
    rng = np.random.default_rng(4 + b)
    G, S, L = 64, 4, (1 << b) - 1
    x = rand_bf16(rng, (400, 128), 3.0)
    res, s, z = per_stage_residuals(x, S, G, oracle, b)
    N = x.shape[0]
    for k in range(S):
        rin = res[k].reshape(N, -1, G)
        rout = res[k + 1].reshape(N, -1, G)
        span = rin.max(-1) - rin.min(-1)
        exact_s = span / L
        slack = np.abs(rin.min(-1) - z[k]) + L * np.abs(exact_s - s[k]) + 1e-6 * (np.abs(rin).max(-1) + 1e-30)
        err = np.abs(rout).max(-1)
        assert np.all(err <= s[k] / 2 + slack + 1e-12), k
        assert np.all(err <= span / (2 * L) + slack + 1e-12), k
    mse = [np.mean(r ** 2) for r in res]
    assert all(mse[k + 1] <= mse[k] for k in range(S)), mse


def test_decode_inverts_encode_within_last_stage_bound(oracle):
    rng = np.random.default_rng(5)
    x = rand_bf16(rng, (200, 128), 1.0)
    C = 8
    cent, ids = oracle.fit(x, C, 3)
    codes, meta = oracle.prq_encode(x, cent, ids, 2, 64)
    out = oracle.decode(codes, meta, ids, cent, 64)
    s, _ = decode_meta(meta)
    bound = np.repeat(s[-1], 64, axis=-1) / 2 + np.abs(f32(x)) * 2 ** -8 + 1e-3 * np.repeat(s[-1], 64, axis=-1)
    assert np.all(np.abs(f32(out) - f32(x)) <= bound + np.abs(f32(x)) * 2 ** -8 + 1e-6)


def test_decode_stage_sum_order(oracle):
    """x_hat = bf16(((c + d1) + d2)), one rounding at the end: an example where
    rounding c + d1 to bf16 first would give a different answer."""
    D, G = 64, 64
    # centroid 1.0; stage 1 contributes 2^-9 on every element, stage 2 2^-9:
    # (1 + 2^-9) + 2^-9 = 1 + 2^-8 -> bf16 tie -> 1.0 (even); rounding after
    # stage 1 would give 1.0 then 1.0 + 2^-9 -> 1.0 as well, so use 3*2^-10.
    cent = np.full((1, D), 0x3F80, np.uint16)
    ids = np.zeros(1, np.int32)
    h = lambda v: int(np.float16(v).view(np.uint16))
    # stage values: q = 0 everywhere, so d = z
    meta = np.array([[[h(0.0) | (h(3 * 2 ** -10) << 16)]], [[h(0.0) | (h(3 * 2 ** -10) << 16)]]], np.uint32)
    codes = np.zeros((2, 1, D // 16), np.uint32)
    out = oracle.decode(codes, meta, ids, cent, G)
    # exact: 1 + 6*2^-10 = 1.005859375 -> nearest bf16 is 1.0078125 (0x3F81)
    assert np.all(out == 0x3F81)


# -------------------------------------------------------- SAS / k-means ---

def exact_sq_dists(x, cent):
    xf = [[bf16_fraction(v) for v in row] for row in x]
    cf = [[bf16_fraction(v) for v in row] for row in cent]
    return [[sum((a - b) ** 2 for a, b in zip(xr, cr)) for cr in cf] for xr in xf]


def test_init_indices_golden(oracle):
    line = [l for l in open(os.path.join(GOLD, "kmeans_init_tiny.txt")) if not l.startswith("#")][0]
    idx = [int(v) for v in line.split()]
    x = np.arange(1560 * 64, dtype=np.int64).reshape(1560, 64).astype(np.uint16)
    x[:, 0] = np.arange(1560)                       # row tag
    cent = oracle.kmeans_init(x, 16)
    assert list(cent[:, 0]) == idx


def test_assign_brute_force_exact(oracle):
    """Exact rational distances on small inputs: the oracle's choice is the
    lowest index among the exact minimisers."""
    rng = np.random.default_rng(6)
    for trial in range(6):
        N, D, C = 40, 16, 7
        x = rand_bf16(rng, (N, D))
        cent = rand_bf16(rng, (C, D))
        if trial % 2:
            cent[4] = cent[1]                       # planted exact tie
            x[:5] = cent[1]                         # distance exactly 0 to both
        ids = oracle.assign(x, cent)
        ex = exact_sq_dists(x, cent)
        for n in range(N):
            m = min(ex[n])
            assert ids[n] == min(j for j in range(C) if ex[n][j] == m)


def test_update_is_exact_mean_rounded(oracle):
    rng = np.random.default_rng(7)
    N, D, C = 90, 8, 5
    x = rand_bf16(rng, (N, D), 3.0)
    ids = rng.integers(0, C - 1, N).astype(np.int32)  # cluster C-1 stays empty
    old = rand_bf16(rng, (C, D))
    new, counts = oracle.update(x, ids, old)
    for j in range(C):
        members = np.nonzero(ids == j)[0]
        assert counts[j] == len(members)
        if len(members) == 0:
            assert np.array_equal(new[j], old[j])
            continue
        for d in range(D):
            mean = sum(bf16_fraction(x[n, d]) for n in members) / len(members)
            assert new[j, d] == round_fraction_to_bf16(mean)


def test_lloyd_sse_non_increasing_and_zero_mean_residuals(oracle):
    wl = WL.TINY
    x = SY.mixture_unit(wl, 0, 0, 1)
    C = wl.clusters
    cent = oracle.kmeans_init(x, C)
    xf = f32(x).astype(np.float64)
    prev = None
    for t in range(6):
        ids = oracle.assign(x, cent)
        sse_before = np.sum((xf - f32(cent).astype(np.float64)[ids]) ** 2)
        cent, counts = oracle.update(x, ids, cent)
        cf = f32(cent).astype(np.float64)
        sse_after = np.sum((xf - cf[ids]) ** 2)
        # update cannot raise the objective by more than the bf16 rounding of the means
        assert sse_after <= sse_before * (1 + 1e-4)
        if prev is not None:
            assert sse_before <= prev * (1 + 1e-4)
        prev = sse_after
        # residuals of each cluster have (nearly) zero mean: |mean - c| <= half a bf16 ulp
        for j in range(C):
            mem = ids == j
            if mem.any():
                mu = xf[mem].mean(0)
                assert np.all(np.abs(mu - cf[j]) <= np.abs(mu) * 2 ** -8 + 1e-30)


def test_separable_mixture_recovers_partition(oracle):
    """Eight well separated centres and C = 8: k-means finds the planted
    partition (up to relabelling)."""
    rng = np.random.default_rng(8)
    D, M, per = 32, 8, 60
    centres = rng.standard_normal((M, D)) * 6.0
    lab = np.repeat(np.arange(M), per)
    rng.shuffle(lab)
    x = SY.f64_to_bf16_bits(centres[lab] + 0.05 * rng.standard_normal((M * per, D)))
    # warm start one point from each true cluster (init from tokens, as the method does)
    first = [int(np.nonzero(lab == m)[0][0]) for m in range(M)]
    cent, ids = oracle.fit(x, M, 4, warm=x[first])
    assert len(set(zip(ids.tolist(), lab.tolist()))) == M
    assert len(set(ids.tolist())) == M


def test_fit_equals_init_plus_lloyd(oracle):
    wl = WL.TINY
    x = SY.mixture_unit(wl, 0, 1, 0)
    cent, ids = oracle.fit(x, wl.clusters, 2)
    c = oracle.kmeans_init(x, wl.clusters)
    for _ in range(2):
        i = oracle.assign(x, c)
        c, _ = oracle.update(x, i, c)
    assert np.array_equal(cent, c) and np.array_equal(ids, i)


# ------------------------------------------------------------- streaming ---

def test_stream_protocol(oracle):
    """Chunk 0 fits cold, chunks 1..k-1 only assign to the cached table, chunk
    k refits warm-started from it (centroid caching, QVG sec. 3)."""
    wl = WL.TINY
    chunk, steps, every = 260, 5, 2
    x = SY.mixture_unit(wl, 0, 0, 0)[: chunk * steps]
    C, T, S, G = 8, 2, 2, 64
    vers, cver, ids, codes, meta = oracle.stream(x, chunk, steps, every, C, T, S, G)
    assert list(cver) == [0, 0, 1, 1, 2] and vers.shape[0] == 3
    c0, i0 = oracle.fit(x[:chunk], C, T)
    assert np.array_equal(vers[0], c0) and np.array_equal(ids[:chunk], i0)
    assert np.array_equal(ids[chunk:2 * chunk], oracle.assign(x[chunk:2 * chunk], c0))
    c1, i2 = oracle.fit(x[2 * chunk:3 * chunk], C, T, warm=c0)
    assert np.array_equal(vers[1], c1) and np.array_equal(ids[2 * chunk:3 * chunk], i2)
    cc, mm = oracle.prq_encode(x[chunk:2 * chunk], c0, ids[chunk:2 * chunk], S, G)
    assert np.array_equal(codes[:, chunk:2 * chunk], cc) and np.array_equal(meta[:, chunk:2 * chunk], mm)


# ----------------------------------------------------------------- sizes ---

def test_bits_per_element_closed_form(oracle):
    for line in open(os.path.join(GOLD, "bits_per_element.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, S, b, G, C, D, N, V, frac = line.split()
        S, b, G, C, D, N, V = map(int, (S, b, G, C, D, N, V))
        want = float(Fraction(frac))
        assert oracle.bits_per_element(S, b, G, C, D, N, V) == pytest.approx(want, rel=1e-12), name


def test_encoded_buffers_match_closed_form(oracle):
    """The bytes the oracle's encoder actually produces (codes, meta, one
    uint8 id per token row, bf16 centroids) equal the closed form."""
    wl = WL.TINY
    x = SY.mixture_unit(wl, 0, 0, 0)
    cent, ids = oracle.fit(x, wl.clusters, 1)
    codes, meta = oracle.prq_encode(x, cent, ids, wl.stages, wl.group_size)
    bits = 8 * (codes.nbytes + meta.nbytes + ids.size * 1 + cent.size * 2)
    want = oracle.bits_per_element(wl.stages, 2, wl.group_size, wl.clusters, wl.head_dim, x.shape[0], 1)
    assert bits / x.size == pytest.approx(want, rel=1e-12)


# ---------------------------------------------------------------- Coral ----

def coral_small(rng, N=20, H=3, D=16, R=4):
    xh = rand_bf16(rng, (N, H * D))
    B = rand_bf16(rng, (H, D, D), 0.25)
    U = rand_bf16(rng, (H * D, R), 0.2)
    W = rand_bf16(rng, (H * D, R), 0.2)
    return xh, B, U, W, H, D, R


def test_coral_block_part_is_block_diagonal_matmul(oracle):
    rng = np.random.default_rng(9)
    xh, B, U, W, H, D, R = coral_small(rng)
    zero = np.zeros_like(U)
    pred = oracle.coral_predict(xh, B, zero, zero, H, D)
    x = f32(xh).astype(np.float64).reshape(-1, H, D)
    Bf = f32(B).astype(np.float64)
    dense = np.zeros((H * D, H * D))
    for h in range(H):
        dense[h * D:(h + 1) * D, h * D:(h + 1) * D] = Bf[h]
    ref = x.reshape(-1, H * D) @ dense.T
    bound = 1e-13 * (np.abs(x.reshape(-1, H * D)) @ np.abs(dense).T + 1)
    assert np.all(np.abs(pred - ref) <= bound)


def test_coral_low_rank_part(oracle):
    rng = np.random.default_rng(10)
    xh, B, U, W, H, D, R = coral_small(rng)
    pred = oracle.coral_predict(xh, np.zeros_like(B), U, W, H, D)
    x = f32(xh).astype(np.float64)
    A = f32(U).astype(np.float64) @ f32(W).astype(np.float64).T      # global rank-R map
    ref = x @ A.T
    assert np.allclose(pred, ref, rtol=1e-12, atol=1e-12)
    # the two parts add: full predictor = block + low rank
    full = oracle.coral_predict(xh, B, U, W, H, D)
    blk = oracle.coral_predict(xh, B, np.zeros_like(U), np.zeros_like(W), H, D)
    assert np.allclose(full, blk + pred, rtol=1e-12, atol=1e-12)


def test_coral_identity_predictor_gives_exact_reconstruction(oracle):
    rng = np.random.default_rng(11)
    xh, B, U, W, H, D, R = coral_small(rng, D=64)
    eye = np.stack([SY.f64_to_bf16_bits(np.eye(D)) for _ in range(H)])
    zero = np.zeros_like(U)
    codes, meta, xn, pred = oracle.coral_encode_layer(xh, xh, eye, zero, zero, H, D, 2, 64)
    s, z = decode_meta(meta)
    assert np.all(s == 0) and np.all(z == 0) and np.all(codes == 0)
    assert np.array_equal(xn, xh)


def test_coral_zero_predictor_is_plain_prq(oracle):
    rng = np.random.default_rng(12)
    N, H, D = 30, 2, 64
    xh = rand_bf16(rng, (N, H * D))
    xn = rand_bf16(rng, (N, H * D))
    B = np.zeros((H, D, D), np.uint16)
    U = np.zeros((H * D, 4), np.uint16)
    codes, meta, xnext, _ = oracle.coral_encode_layer(xh, xn, B, U, U, H, D, 2, 64)
    for h in range(H):
        c, m = oracle.prq_encode(xn.reshape(N, H, D)[:, h], None, None, 2, 64)
        assert np.array_equal(codes[:, h], c) and np.array_equal(meta[:, h], m)
    dec = oracle.coral_decode_layer(xh, codes, meta, B, U, U, H, D, 64)
    assert np.array_equal(dec, xnext)


def test_coral_decode_matches_encoder_reconstruction(oracle):
    rng = np.random.default_rng(13)
    xh, B, U, W, H, D, R = coral_small(rng, D=64)
    xn = rand_bf16(rng, xh.shape)
    codes, meta, xnext, _ = oracle.coral_encode_layer(xh, xn, B, U, W, H, D, 2, 64)
    assert np.array_equal(oracle.coral_decode_layer(xh, codes, meta, B, U, W, H, D, 64), xnext)


# ------------------------------------------------------- generator pins ---

def test_generator_is_deterministic_and_shaped():
    a = SY.mixture_unit(WL.TINY, 0, 0, 0)
    b = SY.mixture_unit(WL.TINY, 0, 0, 0)
    assert np.array_equal(a, b)
    x = f32(a)
    out = SY.outlier_channels(WL.TINY, 0, 0)
    assert len(out) == 2
    rest = np.setdiff1d(np.arange(64), out)
    # outlier channels are about 8x larger
    r = np.abs(x[:, out]).mean() / np.abs(x[:, rest]).mean()
    assert 4 < r < 16
    # sub-range generation agrees with the full unit
    assert np.array_equal(SY.mixture_unit(WL.TINY, 0, 0, 0, 100, 300), a[100:300])


def test_splitmix64_reference_values():
    # SplitMix64 seeded with 0: first outputs of the published generator
    got = [int(v) for v in SY.draws(0, np.arange(3, dtype=np.uint64))]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


# ------------------------------------------------ Coral adapted predictors --

def _fit_inputs(seed, N=400, H=2, D=16, R=4):
    rng = np.random.default_rng(seed)
    xh = SY.f64_to_bf16_bits(rng.standard_normal((N, H * D)))
    y = SY.f64_to_bf16_bits(rng.standard_normal((N, H * D)))
    U = SY.f64_to_bf16_bits(rng.standard_normal((H * D, R)) * 0.2)
    W = SY.f64_to_bf16_bits(rng.standard_normal((H * D, R)) * 0.2)
    return xh, y, U, W, H, D


def test_coral_fit_block_matches_library_solve(oracle):
    """The oracle's Cholesky solve of the ridge normal equations agrees with
    numpy's LU solve (LAPACK) of the same equations, built here in fp64."""
    xh, y, U, W, H, D = _fit_inputs(11)
    B, Z = oracle.coral_fit_block(xh, y, U, W, H, D)
    x = f32(xh).astype(np.float64)
    t = x @ f32(W).astype(np.float64)
    for h in range(H):
        X = x[:, h * D:(h + 1) * D]
        L = t @ f32(U[h * D:(h + 1) * D]).astype(np.float64).T
        Rm = f32(y[:, h * D:(h + 1) * D]).astype(np.float64) - L
        G = X.T @ X
        lam = np.ldexp(np.trace(G) / D, -20)
        Zref = np.linalg.solve(G + lam * np.eye(D), X.T @ Rm)       # [i][o] = B[o][i]
        np.testing.assert_allclose(Z[h], Zref.T, rtol=1e-9, atol=1e-12)
        # B is Z rounded to bf16
        assert np.array_equal(B[h], SY.f64_to_bf16_bits(Zref.T)) or \
            np.max(np.abs(f32(B[h]) - Zref.T) / np.maximum(np.abs(Zref.T), 1e-30)) <= 2.0 ** -8


def test_coral_fit_block_recovers_an_exact_block(oracle):
    """Tokens that are unit vectors e_i (k copies each) and targets y = B x
    with a bf16 block B and no low-rank part: G = k I, so the ridge solution
    is B / (1 + 2^-20), which rounds back to B exactly."""
    rng = np.random.default_rng(12)
    H, D, k = 2, 16, 5
    B0 = SY.f64_to_bf16_bits(rng.standard_normal((H, D, D)))
    N = k * D
    x = np.zeros((N, H * D))
    yv = np.zeros((N, H * D))
    for n in range(N):
        i = n % D
        for h in range(H):
            x[n, h * D + i] = 1.0
            yv[n, h * D:(h + 1) * D] = f32(B0[h][:, i])
    xh, y = SY.f64_to_bf16_bits(x), SY.f64_to_bf16_bits(yv)
    B, Z = oracle.coral_fit_block(xh, y, None, None, H, D)
    assert np.array_equal(B, B0)
    np.testing.assert_allclose(Z, f32(B0).astype(np.float64) / (1 + 2.0 ** -20), rtol=1e-12)


def test_coral_fit_block_zero_input(oracle):
    xh, y, U, W, H, D = _fit_inputs(13)
    xh = np.zeros_like(xh)
    B, Z = oracle.coral_fit_block(xh, y, U, W, H, D)
    assert np.all(B == 0) and np.all(Z == 0)


# ------------------------------------------------ Coral-KV + SAS hybrid ---

def test_f32_to_bf16_rounding_matches_exact_rationals(oracle):
    """The hybrid's vectorised bf16 rounding is round-to-nearest-even: each
    result is the nearest bf16 to the exact fp32 value (ties to an even
    mantissa), checked against exact rationals on random values and on every
    exact tie of one binade."""
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(3000) * np.exp2(rng.integers(-20, 20, 3000))).astype(np.float32)
    ties = (np.float32(1.0) + np.arange(128, dtype=np.float32) * np.float32(2.0 ** -7) + np.float32(2.0 ** -8))
    v = np.concatenate([v, ties, -ties]).astype(np.float32)
    got = oracle.f32_to_bf16_bits(v)
    for x, b in zip(v, got):
        fx = Fraction(float(x))
        # the two bf16 neighbours of x, from truncation and one ulp further from zero
        t = int(np.float32(x).view(np.uint32)) >> 16
        lo, hi = bf16_fraction(t), bf16_fraction(t + 1)
        dl, dh = abs(fx - lo), abs(hi - fx)
        want = t if dl < dh else (t + 1 if dh < dl else (t if t % 2 == 0 else t + 1))
        assert int(b) == want, (x, int(b), want)
    assert np.array_equal(oracle.bf16_bits_to_f32(got[:10]).view(np.uint32) >> 16, got[:10].astype(np.uint32))


def test_coral_sas_zero_prediction_is_plain_qvg(oracle):
    """With no previous layer the prediction is 0, so the residual is x_next
    itself (exact in bf16), and the hybrid must reduce to the plain SAS + PRQ
    path of every head: same centroids, ids, codes, meta, and x_hat equal to
    the plain decode (0 + r_hat is exact)."""
    rng = np.random.default_rng(8)
    H, D, N, C, T, S, G = 2, 128, 300, 8, 3, 2, 64
    x = SY.f64_to_bf16_bits(rng.standard_normal((N, H * D)))
    cent, ids, codes, meta, xh, pred = oracle.coral_sas_layer(None, x, None, None, None, H, D, C, T, S, G)
    assert np.all(pred == 0)
    for h in range(H):
        xh_h = np.ascontiguousarray(x[:, h * D:(h + 1) * D])
        oc, oi = oracle.fit(xh_h, C, T)
        rc, rm = oracle.prq_encode(xh_h, oc, oi, S, G)
        np.testing.assert_array_equal(cent[h], oc)
        np.testing.assert_array_equal(ids[h], oi)
        np.testing.assert_array_equal(codes[:, h], rc)
        np.testing.assert_array_equal(meta[:, h], rm)
        np.testing.assert_array_equal(xh[:, h * D:(h + 1) * D], oracle.decode(rc, rm, oi, oc, G))


def test_coral_sas_perfect_prediction_reconstructs_exactly(oracle):
    """A prediction equal to x_next leaves a zero residual: every group is
    constant (scale 0), the decoded residual is 0, and x_hat = bf16(pred + 0)
    = x_next exactly."""
    rng = np.random.default_rng(9)
    H, D, N, C, T, S, G = 2, 128, 200, 4, 2, 2, 64
    x = SY.f64_to_bf16_bits(rng.standard_normal((N, H * D)))
    pred = oracle.bf16_bits_to_f32(x)
    cent, ids, codes, meta, xh, _ = oracle.coral_sas_layer(None, x, None, None, None, H, D, C, T, S, G, pred_in=pred)
    np.testing.assert_array_equal(xh, x)
    assert np.all(cent == 0)
    assert np.all(meta & 0xFFFF == 0)                     # every stage scale is 0


def test_coral_sas_residual_and_reconstruction_arithmetic(oracle):
    """The residual is the fp32 difference rounded once to bf16, and the
    reconstruction adds the decoded residual to the fp32 prediction: checked
    element by element against exact rationals for a random prediction."""
    rng = np.random.default_rng(10)
    H, D, N, C, T, S, G = 1, 128, 64, 4, 2, 2, 64
    x = SY.f64_to_bf16_bits(rng.standard_normal((N, H * D)))
    pred = (rng.standard_normal((N, H * D)) * 0.5).astype(np.float32)
    cent, ids, codes, meta, xh, _ = oracle.coral_sas_layer(None, x, None, None, None, H, D, C, T, S, G, pred_in=pred)
    rhat = oracle.decode(codes[:, 0], meta[:, 0], ids[0], cent[0], G)
    for n in range(0, N, 7):
        for i in range(0, D, 11):
            # reconstruction: RN_bf16(RN_f32(pred + r_hat)) from exact rationals
            s = np.float32(Fraction(float(pred[n, i])) + bf16_fraction(rhat[n, i]))
            t = int(np.float32(s).view(np.uint32)) >> 16
            lo, hi = bf16_fraction(t), bf16_fraction(t + 1)
            fs = Fraction(float(s))
            want = t if abs(fs - lo) < abs(hi - fs) else (t + 1 if abs(hi - fs) < abs(fs - lo) else (t if t % 2 == 0 else t + 1))
            assert int(xh[n, i]) == want
    # the residual enters with its sign and scale: two 2-bit stages leave at
    # most span/18 of a group's residual, so the reconstruction error is far
    # below the prediction error (a flipped or rescaled residual is not)
    xf, hf = oracle.bf16_bits_to_f32(x).astype(np.float64), oracle.bf16_bits_to_f32(xh).astype(np.float64)
    assert np.max(np.abs(hf - xf)) <= 0.25 * np.max(np.abs(xf - pred)) + 2.0 ** -6


# ------------------------------------------- attention over the decoded cache --
# Pins of oracle.attention (Quant VideoGen explainer, sec. 3: dequantisation
# fused into the consumer; 33-method Self-Forcing KV-cache study, abstract:
# attention over the rebuilt keys and values).

def _bf16_rows(rng, n, d, scale=1.0):
    return SY.f64_to_bf16_bits(scale * rng.standard_normal((n, d)))


def test_attention_matches_torch_sdpa_in_fp64(oracle):
    """Against torch's scaled-dot-product attention (a library routine) run in
    fp64 on the CPU, with the scale passed explicitly."""
    import torch
    rng = np.random.default_rng(21)
    for nq, n, d, scale in ((5, 7, 64, 0.125), (33, 300, 128, 128 ** -0.5), (1, 1, 64, 2.0)):
        q, k, v = _bf16_rows(rng, nq, d), _bf16_rows(rng, n, d), _bf16_rows(rng, n, d)
        o = oracle.attention(q, k, v, np.float32(scale))
        t = [torch.from_numpy(SY.bf16_bits_to_f32(a).astype(np.float64))[None] for a in (q, k, v)]
        ref = torch.nn.functional.scaled_dot_product_attention(*t, scale=float(np.float32(scale)))[0].numpy()
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_attention_closed_forms(oracle):
    """q = 0 gives equal weights, so every output row is the mean of the
    value rows; one key gives that key's value row exactly; two keys whose
    scores differ by ln 3 weigh their values 1/4 and 3/4."""
    rng = np.random.default_rng(22)
    n, d = 40, 64
    k, v = _bf16_rows(rng, n, d), _bf16_rows(rng, n, d)
    vf = SY.bf16_bits_to_f32(v).astype(np.float64)
    o = oracle.attention(np.zeros((3, d), np.uint16), k, v, 0.5)
    np.testing.assert_allclose(o, np.broadcast_to(vf.mean(axis=0), o.shape), rtol=0, atol=1e-13)
    o1 = oracle.attention(_bf16_rows(rng, 4, d), k[:1], v[:1], 0.3)
    np.testing.assert_array_equal(o1, np.broadcast_to(vf[0], o1.shape))
    # q = e_0, k_0 = 0, k_1 = e_0: scores 0 and `scale`, with scale = ln 3 in fp32
    q = np.zeros((1, d), np.uint16); q[0, 0] = 0x3F80          # 1.0
    k2 = np.zeros((2, d), np.uint16); k2[1, 0] = 0x3F80
    sc = np.float32(np.log(3.0))
    w1 = 3.0 * np.exp(float(sc) - np.log(3.0))                  # 3 up to the fp32 rounding of ln 3
    expect = (vf[0] + w1 * vf[1]) / (1.0 + w1)
    np.testing.assert_allclose(oracle.attention(q, k2, v[:2], sc)[0], expect, rtol=0, atol=1e-14)
    assert abs(w1 - 3.0) < 1e-6


def test_attention_invariances(oracle):
    """Permuting the (key, value) rows together leaves the output unchanged;
    adding the same vector to every value row adds it to every output row
    (the weights sum to 1); a key whose score leads by 800 takes all weight."""
    rng = np.random.default_rng(23)
    nq, n, d = 6, 50, 64
    q, k, v = _bf16_rows(rng, nq, d), _bf16_rows(rng, n, d), _bf16_rows(rng, n, d)
    o = oracle.attention(q, k, v, 0.125)
    perm = rng.permutation(n)
    np.testing.assert_allclose(oracle.attention(q, k[perm], v[perm], 0.125), o, rtol=0, atol=1e-13)
    # multiples of 1/8 below 2 stay exact in bf16 after adding 2.0
    vs = SY.f64_to_bf16_bits(rng.integers(0, 16, (n, d)) / 8.0)
    v2 = SY.f64_to_bf16_bits(SY.bf16_bits_to_f32(vs).astype(np.float64) + 2.0)
    np.testing.assert_allclose(oracle.attention(q, k, v2, 0.125), oracle.attention(q, k, vs, 0.125) + 2.0,
                               rtol=0, atol=1e-12)
    qd = np.zeros((1, d), np.uint16); qd[0, 3] = 0x3F80
    kd = np.zeros((n, d), np.uint16); kd[17, 3] = 0x4448         # 800.0
    vf = SY.bf16_bits_to_f32(v).astype(np.float64)
    np.testing.assert_allclose(oracle.attention(qd, kd, v, 1.0)[0], vf[17], rtol=0, atol=1e-300)
