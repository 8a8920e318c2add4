"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

Each check below ties the oracle to something other than itself: a closed
form, a hand-enumerated case, an independent library routine (numpy's FFT,
which the oracle does not use), brute force over all codes, an inequality
that must hold, or a number printed on one of the pages
(``tests/golden/pages_memory.json``, each entry with its citation).  The
mutation tests at the end plant plausible mistakes in the oracle and check
that some pin fails, so the pins are known to be sharp.
"""

import cmath
import json
import math
import os

import numpy as np
import pytest

from oracle import srft_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DIMS = (4, 8, 16, 32, 64, 128, 256)
ODD_DIMS = (6, 12, 80, 96, 192)  # even, not powers of two (reading 10)
POW2 = DIMS


# ---------------------------------------------------------------- sign vector

def check_splitmix_vectors(o):
    # First three outputs of the reference splitmix64 generator seeded with 0
    # (Vigna's splitmix64.c; the same sequence as Java's SplittableRandom(0)).
    assert o.splitmix64_stream(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_published_outputs():
    check_splitmix_vectors(O)


def test_sign_vector_is_bit63_of_the_stream():
    words = O.splitmix64_stream(123, 256)
    s = O.sign_vector(256, 123)
    assert set(np.unique(s)) <= {-1.0, 1.0}
    for i, w in enumerate(words):
        assert s[i] == (-1.0 if w >= 1 << 63 else 1.0)
    # roughly balanced (a fixed-point check that bit 63 is a fair coin here)
    assert 96 <= int((s < 0).sum()) <= 160
    # the same seed gives the same prefix at every d
    assert np.array_equal(O.sign_vector(64, 123), s[:64])


# ---------------------------------------------------------------- transform

def check_unitarity(o, d, seed=7):
    R = o.srft_matrix(d, seed)
    assert np.abs(R.T @ R - np.eye(d)).max() < 1e-12
    rng = np.random.default_rng(d)
    x, y = rng.standard_normal((2, d))
    px, py = o.srft_forward(x, seed), o.srft_forward(y, seed)
    assert abs(np.linalg.norm(px) - np.linalg.norm(x)) < 1e-12 * np.linalg.norm(x)
    assert abs(px @ py - x @ y) < 1e-12 * np.linalg.norm(x) * np.linalg.norm(y)


@pytest.mark.parametrize("d", DIMS + ODD_DIMS)
def test_unitarity(d):
    check_unitarity(O, d)


def check_basis_closed_form(o, d, seed=11):
    """R e_j = s_j [1/sqrt d, (-1)^j/sqrt d, sqrt(2/d) cos(2 pi jk/d), -sqrt(2/d) sin(2 pi jk/d), ...]."""
    s = o.sign_vector(d, seed)
    R = o.srft_matrix(d, seed)
    for j in range(d):
        col = [1 / math.sqrt(d), (-1) ** j / math.sqrt(d)]
        for k in range(1, d // 2):
            a = 2 * math.pi * j * k / d
            col += [math.sqrt(2 / d) * math.cos(a), -math.sqrt(2 / d) * math.sin(a)]
        assert np.abs(R[:, j] - s[j] * np.array(col)).max() < 1e-13


@pytest.mark.parametrize("d", (4, 8, 16, 64, 6, 12, 96, 192))
def test_basis_vectors_closed_form(d):
    check_basis_closed_form(O, d)


def test_d4_by_hand():
    x = np.array([0.3, -1.7, 2.5, 0.25])
    s = O.sign_vector(4, 5)
    u0, u1, u2, u3 = s * x
    y0 = (u0 + u1 + u2 + u3) / 2
    y2 = (u0 - u1 + u2 - u3) / 2
    y1 = complex(u0 - u2, -(u1 - u3)) / 2
    want = [y0, y2, math.sqrt(2) * y1.real, math.sqrt(2) * y1.imag]
    assert np.abs(O.srft_forward(x, 5) - want).max() < 1e-14


def test_d8_brute_force_complex_sums():
    """Every entry of the 8x8 R from an explicit complex sum, written out in pure Python."""
    d, seed = 8, 2
    s = O.sign_vector(d, seed)
    R = O.srft_matrix(d, seed)
    for j in range(d):
        u = [0.0] * d
        u[j] = s[j]
        y = [sum(u[n] * cmath.exp(-2j * math.pi * n * k / d) for n in range(d)) / math.sqrt(d)
             for k in range(d // 2 + 1)]
        col = [y[0].real, y[4].real]
        for k in range(1, 4):
            col += [math.sqrt(2) * y[k].real, math.sqrt(2) * y[k].imag]
        assert np.abs(R[:, j] - col).max() < 1e-14


def check_matches_numpy_fft(o, d, seed=3):
    rng = np.random.default_rng(100 + d)
    x = rng.standard_normal((6, d))
    y = np.fft.rfft(x * o.sign_vector(d, seed), axis=-1, norm="ortho")
    half = d // 2
    want = np.empty_like(x)
    want[:, 0], want[:, 1] = y[:, 0].real, y[:, half].real
    want[:, 2::2] = math.sqrt(2) * y[:, 1:half].real
    want[:, 3::2] = math.sqrt(2) * y[:, 1:half].imag
    assert np.abs(o.srft_forward(x, seed) - want).max() < 1e-12


@pytest.mark.parametrize("d", DIMS + ODD_DIMS)
def test_matches_numpy_fft(d):
    check_matches_numpy_fft(O, d)


@pytest.mark.parametrize("d", DIMS + ODD_DIMS)
def test_exact_round_trip_and_numpy_inverse(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((5, d))
    p = O.srft_forward(x, 9)
    assert np.abs(O.srft_inverse(p, 9) - x).max() < 1e-12
    # the inverse on its own, against numpy's inverse real FFT
    half = d // 2
    y = np.zeros((5, half + 1), dtype=complex)
    y[:, 0], y[:, half] = p[:, 0], p[:, 1]
    y[:, 1:half] = (p[:, 2::2] + 1j * p[:, 3::2]) / math.sqrt(2)
    u = np.fft.irfft(y, n=d, axis=-1, norm="ortho")
    assert np.abs(O.srft_inverse(p, 9) - u * O.sign_vector(d, 9)).max() < 1e-12


# ---------------------------------------------------------------- quantiser

def _brute_codes(z, scale, Q):
    cands = np.arange(-Q, Q + 1)
    return np.array([cands[np.argmin(np.abs(zi - cands * scale))] for zi in z])


@pytest.mark.parametrize("bits", (4, 8))
@pytest.mark.parametrize("d,g", ((8, 4), (8, 8), (16, 16), (16, 8)))
def test_quantiser_brute_force(bits, d, g):
    rng = np.random.default_rng(bits * 100 + d + g)
    Q = O.qmax(bits)
    for _ in range(50):
        z = rng.standard_normal(d) * rng.uniform(0.1, 10)
        q, scale, r = O.quantize_groups(z, bits, g)
        for j in range(d // g):
            sl = slice(j * g, (j + 1) * g)
            A = np.abs(z[sl]).max()
            assert scale[j] == pytest.approx(A / Q, rel=1e-15)
            frac = np.abs(r[sl] - np.floor(r[sl]) - 0.5)
            ok = frac > 1e-9  # ties are decided by the tie rule, checked separately
            assert np.array_equal(q[sl][ok], _brute_codes(z[sl], scale[j], Q)[ok])
            # the absmax coordinate maps to +-Q
            i = np.argmax(np.abs(z[sl]))
            assert abs(q[sl][i]) == Q and np.sign(q[sl][i]) == np.sign(z[sl][i])


def test_quantiser_ties_round_half_even_and_symmetric_range():
    z = np.array([7.0, 2.5, -2.5, 0.5, -0.5, 1.5, 3.5, -7.0])  # A = 7, Q = 7 -> scale 1
    q, scale, _ = O.quantize_groups(z, 4, 8)
    assert scale[0] == 1.0
    assert q.tolist() == [7, 2, -2, 0, 0, 2, 4, -7]
    z8 = np.array([-127.0, 126.5, 0.0, 1.0])
    q8, s8, _ = O.quantize_groups(z8, 8, 4)
    assert s8[0] == 1.0 and q8.tolist() == [-127, 126, 0, 1]


def test_zero_vector_and_single_spike():
    for bits in (4, 8):
        out = O.srft_kv_quantize(np.zeros((3, 64)), None, bits, 16, 1)
        assert not out["scales"].any() and not out["codes"].any()
        # x = a R^{-1} e_i has exactly one nonzero rotated coordinate
        for i in (0, 1, 5, 63):
            e = np.zeros(64)
            e[i] = 3.25
            x = O.srft_inverse(e, 1)
            enc = O.srft_kv_quantize(x, None, bits, 16, 1)
            j = i // 16
            want = np.zeros(16, dtype=np.int64)
            want[i % 16] = O.qmax(bits)
            assert np.array_equal(enc["q"][16 * j : 16 * j + 16], want)
            assert enc["scales"][j] == pytest.approx(3.25 / O.qmax(bits), rel=1e-14)
            # the other groups only hold rounding residue of the fp64 transform
            assert np.delete(enc["scales"], j).max() < 1e-14


def check_packing(o):
    assert o.pack_codes(np.array([-7, 7]), 4).tolist() == [0x79]
    assert o.pack_codes(np.array([-1, 0, 3, -4]), 4).tolist() == [0x0F, 0xC3]
    assert o.pack_codes(np.array([-127, 127, -1, 0]), 8).tolist() == [0x81, 0x7F, 0xFF, 0x00]


def test_nibble_and_byte_packing_by_hand():
    check_packing(O)
    q = np.random.default_rng(0).integers(-7, 8, (4, 32))
    assert np.array_equal(O.unpack_codes(O.pack_codes(q, 4), 4), q)
    q8 = np.random.default_rng(1).integers(-127, 128, (4, 32))
    assert np.array_equal(O.unpack_codes(O.pack_codes(q8, 8), 8), q8)


@pytest.mark.parametrize("bits", (4, 8))
def test_dequantisation_error_bounds(bits):
    rng = np.random.default_rng(bits)
    d, g = 128, 16
    x = rng.standard_normal((20, d))
    x[:, 5] *= 40
    lam = np.exp(0.5 * rng.standard_normal(d))
    enc = O.srft_kv_quantize(x, lam, bits, g, 3)
    zhat = O.unpack_codes(enc["codes"], bits) * np.repeat(enc["scales"], g, axis=-1)
    step = np.repeat(enc["scales"], g, axis=-1)
    assert np.all(np.abs(zhat - enc["z"]) <= step / 2 * (1 + 1e-12))
    xhat = O.srft_kv_dequantize(enc["codes"], enc["scales"], lam, bits, g, 3)
    bound = np.linalg.norm(step / (2 * lam), axis=-1)
    assert np.all(np.linalg.norm(xhat - x, axis=-1) <= bound * (1 + 1e-12))


def test_rotation_spreads_an_outlier_channel():
    """A single large channel is spread over all rotated coordinates (page claim, in math form)."""
    d = 128
    x = np.zeros(d)
    x[17] = 50.0
    p = O.srft_forward(x, 4)
    assert np.abs(p).max() <= 50.0 * math.sqrt(2 / d) * (1 + 1e-12)


# ---------------------------------------------------------------- attention

def test_attention_single_token_and_equal_keys():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((2, 4, 8))
    v = rng.standard_normal((2, 5, 2, 8))
    k1 = rng.standard_normal((2, 1, 2, 8))
    o1 = O.decode_attention(q, k1, v[:, :1])
    for h in range(4):
        assert np.abs(o1[:, h] - v[:, 0, h // 2]).max() < 1e-12
    k_eq = np.repeat(k1, 5, axis=1)
    oe = O.decode_attention(q, k_eq, v)
    for h in range(4):
        assert np.abs(oe[:, h] - v[:, :, h // 2].mean(axis=1)).max() < 1e-12


def test_attention_tiny_case_by_hand():
    """d=8, T=3, one head, softmax written out with math.exp."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 1, 8))
    k = rng.standard_normal((1, 3, 1, 8))
    v = rng.standard_normal((1, 3, 1, 8))
    sc = 0.3
    s = [sc * sum(q[0, 0, i] * k[0, t, 0, i] for i in range(8)) for t in range(3)]
    e = [math.exp(x) for x in s]
    want = [sum(e[t] * v[0, t, 0, i] for t in range(3)) / sum(e) for i in range(8)]
    assert np.abs(O.decode_attention(q, k, v, sm_scale=sc)[0, 0] - want).max() < 1e-12
    # default scale is 1/sqrt(d)
    s2 = O.decode_attention(q, k, v)
    assert np.abs(s2 - O.decode_attention(q, k, v, sm_scale=1 / math.sqrt(8))).max() == 0


def check_gqa_and_lengths(o):
    rng = np.random.default_rng(9)
    B, Hq, Hkv, T, d = 2, 6, 3, 7, 8
    q = rng.standard_normal((B, Hq, d))
    k = rng.standard_normal((B, T, Hkv, d))
    v = rng.standard_normal((B, T, Hkv, d))
    L = [7, 3]
    out = o.decode_attention(q, k, v, seq_lens=L)
    for b in range(B):
        for h in range(Hq):
            kv = h // (Hq // Hkv)  # consecutive query heads share a kv head
            s = k[b, : L[b], kv] @ q[b, h] / math.sqrt(d)
            w = np.exp(s - s.max())
            assert np.abs(out[b, h] - (w @ v[b, : L[b], kv]) / w.sum()).max() < 1e-12
    # tokens past the sequence length do not matter; a zero length gives zeros
    k2 = k.copy()
    k2[1, 3:] = 1e3
    assert np.abs(o.decode_attention(q, k2, v, seq_lens=L) - out).max() == 0
    assert not o.decode_attention(q, k, v, seq_lens=[0, 0]).any()


def test_gqa_mapping_and_sequence_lengths():
    check_gqa_and_lengths(O)


def test_rotated_domain_scores_equal_unrotated():
    """q . k_hat == SRFT(q) . (z_hat / lambda): the identity the GPU kernel relies on."""
    rng = np.random.default_rng(2)
    d, g = 128, 16
    k = rng.standard_normal((16, d))
    lam = np.exp(0.5 * rng.standard_normal(d))
    q = rng.standard_normal(d)
    enc = O.srft_kv_quantize(k, lam, 4, g, 8)
    khat = O.srft_kv_dequantize(enc["codes"], enc["scales"], lam, 4, g, 8)
    prot = O.dequantize_rotated(enc["codes"], enc["scales"], lam, 4, g)
    assert np.abs(khat @ q - prot @ O.srft_forward(q, 8)).max() < 1e-12


# ---------------------------------------------------------------- page numbers

def _golden():
    with open(os.path.join(GOLDEN, "pages_memory.json")) as f:
        return json.load(f)


def test_kv_memory_formula_against_page_examples():
    for c in _golden()["kv_memory_formula"]["cases"]:
        b = O.kv_bytes(c["layers"], c["kv_heads"], c["head_dim"], c["seq_len"], c["dtype_bytes"])
        assert b == 2 * c["layers"] * c["kv_heads"] * c["head_dim"] * c["seq_len"] * c["dtype_bytes"]
        assert b / 2**30 == c["approx_gb"]  # 6 GiB and 12 GiB exactly


def test_kvsplit_table_ratios():
    g = _golden()["kvsplit_8k_table"]
    L, H, d, T = 1, 1, 128, 8192  # the ratios do not depend on the (unnamed) model shape
    fp16 = O.kv_bytes(L, H, d, T, 2)
    for row in g["rows"]:
        packed = O.packed_kv_bytes(L, H, d, T, row["bits_k"], row["bits_v"], group=32, scale_bytes=2)
        assert packed / fp16 == row["mb"] / g["fp16_mb"]
        assert round(100 * (1 - packed / fp16)) == row["saving_pct"]


def test_kvsplit_k8v4_formula_and_compression_ratio():
    gl = _golden()
    L, H, d, T = 32, 8, 128, 8192
    no_scales = O.packed_kv_bytes(L, H, d, T, 8, 4, group=d, scale_bytes=0)
    assert no_scales == L * H * d * T * gl["kvsplit_k8v4_formula"]["k8v4_bytes_per_element_pair"]
    ratio = O.kv_bytes(1, 1, 128, 1, 2) / O.packed_kv_bytes(1, 1, 128, 1, 4, 4, group=32, scale_bytes=2)
    assert round(ratio, 2) == gl["compression"]["max_ratio"]


def test_non_power_of_two_d6_by_hand():
    """d = 6: the 3 + 1 bins of a real length-6 DFT, packed, from explicit complex sums."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal(6)
    s = O.sign_vector(6, 2)
    u = x * s
    y = [sum(u[n] * cmath.exp(-2j * math.pi * n * k / 6) for n in range(6)) / math.sqrt(6) for k in range(4)]
    want = [y[0].real, y[3].real, math.sqrt(2) * y[1].real, math.sqrt(2) * y[1].imag, math.sqrt(2) * y[2].real,
            math.sqrt(2) * y[2].imag]
    assert np.abs(O.srft_forward(x, 2) - np.array(want)).max() < 1e-13


def test_hadamard_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        O.hadamard_matrix(96)


# ---------------------------------------------------------------- Hadamard variant (SRHT)

def check_hadamard_matches_scipy(o, d):
    # scipy builds H by the Sylvester recursion, independently of the popcount form
    scipy_linalg = pytest.importorskip("scipy.linalg")
    assert np.array_equal(o.hadamard_matrix(d), scipy_linalg.hadamard(d).astype(np.float64))


@pytest.mark.parametrize("d", POW2)
def test_hadamard_matches_scipy(d):
    check_hadamard_matches_scipy(O, d)


def test_hadamard_d4_by_hand_and_sylvester_recursion():
    h4 = np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]], dtype=np.float64)
    assert np.array_equal(O.hadamard_matrix(4), h4)
    for d in (4, 8, 16, 32):
        h = O.hadamard_matrix(d)
        assert np.array_equal(O.hadamard_matrix(2 * d), np.block([[h, h], [h, -h]]))


@pytest.mark.parametrize("d", DIMS)
def test_srht_orthogonal_and_round_trip(d):
    R = O.srht_matrix(d, 7)
    assert np.abs(R.T @ R - np.eye(d)).max() < 1e-12
    rng = np.random.default_rng(d)
    x = rng.standard_normal((5, d))
    assert np.abs(O.srht_inverse(O.srht_forward(x, 7), 7) - x).max() < 1e-12
    assert np.abs(np.linalg.norm(O.srht_forward(x, 7), axis=-1) - np.linalg.norm(x, axis=-1)).max() < 1e-12


def _fwht(u):
    """Fast Walsh-Hadamard transform by in-place butterflies (O(d log d)), written here from the
    definition of the Sylvester recursion; independent of the oracle's matrix."""
    u = np.array(u, dtype=np.float64)
    h = 1
    while h < u.shape[-1]:
        for i in range(0, u.shape[-1], 2 * h):
            a = u[..., i:i + h].copy()
            b = u[..., i + h:i + 2 * h].copy()
            u[..., i:i + h], u[..., i + h:i + 2 * h] = a + b, a - b
        h *= 2
    return u


@pytest.mark.parametrize("d", DIMS)
def test_srht_equals_signed_fast_wht(d):
    rng = np.random.default_rng(100 + d)
    x = rng.standard_normal((3, d))
    s = O.sign_vector(d, 11)
    assert np.abs(O.srht_forward(x, 11) - _fwht(x * s) / math.sqrt(d)).max() < 1e-12


def test_srht_quantiser_and_attention_identity():
    rng = np.random.default_rng(5)
    d, g = 16, 8
    x = rng.standard_normal((4, d)).astype(np.float16).astype(np.float64)
    enc = O.srft_kv_quantize(x, None, 4, g, 9, transform="srht")
    assert np.abs(enc["z"] - _fwht(x * O.sign_vector(d, 9)) / math.sqrt(d)).max() < 1e-12
    # brute force: every code is the nearest of the 2Q+1 levels of its group's scale
    sc = np.repeat(enc["scales"], g, axis=-1)
    levels = np.arange(-7, 8)
    best = levels[np.argmin(np.abs(enc["z"][..., None] - levels * sc[..., None]), axis=-1)]
    assert np.array_equal(enc["q"], best)
    # the dequantised cache is the SRHT inverse of q * scale, and q . k_hat is preserved by the rotation
    xhat = O.srft_kv_dequantize(enc["codes"], enc["scales"], None, 4, g, 9, transform="srht")
    assert np.abs(_fwht(xhat * O.sign_vector(d, 9)) / math.sqrt(d) - enc["q"] * sc).max() < 1e-12
    q = rng.standard_normal(d)
    assert np.abs(xhat @ q - (enc["q"] * sc) @ O.srht_forward(q, 9)).max() < 1e-12


# ---------------------------------------------------------------- lighter scale planes (fp16, e8m0)

def _all_fp16_values():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = bits.view(np.float16).astype(np.float64)
    ok = np.isfinite(v)
    return v[ok], bits[ok]


def check_fp16_scale_rounding(o):
    """Brute force over every finite fp16: the stored scale is the nearest one to A/Q (ties to the even bit
    pattern), saturating at 65504."""
    vals, bits = _all_fp16_values()
    rng = np.random.default_rng(3)
    targets = np.concatenate([rng.lognormal(0.0, 4.0, 300), vals[(vals > 0) & (vals < 70000)][::997] *
                              (1 + 2.0**-12), [1e6, 65504.0, 65519.0, 6e-8, 1e-9]])
    got = o.fp16_round(targets)
    for t, g in zip(targets, got):
        dist = np.abs(vals - t)
        near = np.flatnonzero(dist == dist.min())
        if len(near) > 1:  # a tie: the even bit pattern wins
            near = near[(bits[near] & 1) == 0]
        want = min(vals[near[0]], 65504.0)
        assert g == want, (t, g, want)


def test_fp16_scale_is_nearest_fp16():
    check_fp16_scale_rounding(O)


def check_e8m0_scale(o):
    rng = np.random.default_rng(4)
    a = np.concatenate([rng.lognormal(0.0, 6.0, 500), np.ldexp(1.0, np.arange(-20, 21)).astype(np.float64)])
    v, raw = o.store_scales(a, "e8m0")
    assert np.all(v >= a) and np.all(v / 2 < a)  # the smallest power of two not below A/Q
    assert np.array_equal(np.log2(v), raw.astype(np.int64) - 127)
    assert np.array_equal(o.decode_scales(raw, "e8m0"), v)
    p2 = np.ldexp(1.0, np.arange(-20, 21))
    assert np.array_equal(o.store_scales(p2, "e8m0")[0], p2)  # exact powers of two map to themselves


def test_e8m0_scale_is_smallest_power_of_two_above():
    check_e8m0_scale(O)


@pytest.mark.parametrize("fmt", ("fp16", "e8m0"))
@pytest.mark.parametrize("bits", (4, 8))
def test_codes_against_the_stored_scale(fmt, bits):
    rng = np.random.default_rng(bits)
    d, g = 32, 16
    x = (rng.standard_normal((6, d)) * 3).astype(np.float16).astype(np.float64)
    enc = O.srft_kv_quantize(x, None, bits, g, 5, scale_format=fmt)
    Q = O.qmax(bits)
    sc = np.repeat(enc["scales"], g, axis=-1)
    levels = np.arange(-Q, Q + 1)
    best = levels[np.argmin(np.abs(enc["z"][..., None] - levels * sc[..., None]), axis=-1)]
    assert np.array_equal(enc["q"], best)
    assert np.array_equal(O.decode_scales(enc["scales_raw"], fmt), enc["scales"])
    if fmt == "e8m0":  # no code needs clamping: |z| / scale <= Q
        assert np.all(np.abs(enc["r"]) <= Q)
    # zero groups store 0 and codes 0
    z0 = O.srft_kv_quantize(np.zeros((1, d)), None, bits, g, 5, scale_format=fmt)
    assert not z0["scales"].any() and not z0["q"].any() and not np.asarray(z0["scales_raw"]).any()


def test_lighter_scale_planes_give_the_pages_compression():
    # [WQF] Key results, memory efficiency: 3.0x to 3.56x persistent compression (tests/golden/pages_memory.json)
    with open(os.path.join(GOLDEN, "pages_memory.json")) as f:
        gl = json.load(f)
    fp16_vec = 2 * 128
    assert round(fp16_vec / O.packed_vector_bytes(128, 4, 16, O.SCALE_BYTES["e8m0"]), 2) == gl["compression"]["max_ratio"]
    assert fp16_vec / O.packed_vector_bytes(128, 4, 16, O.SCALE_BYTES["fp16"]) == pytest.approx(3.2)
    assert fp16_vec / O.packed_vector_bytes(128, 4, 16, O.SCALE_BYTES["fp32"]) == pytest.approx(2.67, abs=0.005)


# ---------------------------------------------------------------- mutation tests

class _Mutant:
    """The oracle module with one function replaced."""

    def __init__(self, **repl):
        self.__dict__.update({k: getattr(O, k) for k in dir(O) if not k.startswith("__")})
        self.__dict__.update(repl)


def _mutant_forward(pack=None, dft=None, sign=None):
    pack = pack or O.hermitian_pack
    dft = dft or O.dft_half_matrix
    sign = sign or O.sign_vector

    def fwd(x, seed):
        x = np.asarray(x, dtype=np.float64)
        d = x.shape[-1]
        return pack((x * sign(d, seed)) @ dft(d).T)

    def mat(d, seed):
        return fwd(np.eye(d), seed).T

    return _Mutant(srft_forward=fwd, srft_matrix=mat)


def test_mutant_wrong_dft_sign_is_caught():
    m = _mutant_forward(dft=lambda d: np.conj(O.dft_half_matrix(d)))
    check_unitarity(m, 16)  # still orthogonal ...
    with pytest.raises(AssertionError):
        check_matches_numpy_fft(m, 16)  # ... but not the DFT
    with pytest.raises(AssertionError):
        check_basis_closed_form(m, 16)


def test_mutant_dropped_sqrt2_is_caught():
    def bad_pack(y):
        p = O.hermitian_pack(y)
        p[..., 2:] /= math.sqrt(2)
        return p

    with pytest.raises(AssertionError):
        check_unitarity(_mutant_forward(pack=bad_pack), 16)


def test_mutant_swapped_re_im_is_caught():
    def bad_pack(y):
        p = O.hermitian_pack(y)
        p[..., 2::2], p[..., 3::2] = p[..., 3::2].copy(), p[..., 2::2].copy()
        return p

    m = _mutant_forward(pack=bad_pack)
    with pytest.raises(AssertionError):
        check_matches_numpy_fft(m, 16)


def test_mutant_swapped_nibbles_is_caught():
    def bad_pack_codes(q, bits):
        b = O.pack_codes(q, bits)
        return ((b >> 4) | (b << 4)) & 0xFF if bits == 4 else b

    with pytest.raises(AssertionError):
        check_packing(_Mutant(pack_codes=bad_pack_codes))


def test_mutant_gqa_modulo_mapping_is_caught():
    def bad_attention(q, k, v, seq_lens=None, sm_scale=None):
        # maps query head h to kv head h % Hkv instead of h // (Hq / Hkv)
        B, Hq, d = q.shape
        Hkv = k.shape[2]
        perm = [h % Hkv for h in range(Hq)]
        kk = np.stack([k[:, :, p] for p in perm], axis=2)
        vv = np.stack([v[:, :, p] for p in perm], axis=2)
        return O.decode_attention(q, kk, vv, seq_lens, sm_scale)

    with pytest.raises(AssertionError):
        check_gqa_and_lengths(_Mutant(decode_attention=bad_attention))


def test_mutant_wrong_splitmix_constant_is_caught():
    def bad_stream(seed, n):
        return [O.splitmix64((seed + i * O.SPLITMIX_GAMMA) & O.MASK64) for i in range(n)]

    with pytest.raises(AssertionError):
        check_splitmix_vectors(_Mutant(splitmix64_stream=bad_stream))


def test_mutant_hadamard_wrong_index_rule_is_caught():
    def bad_hadamard(d):
        i = np.arange(d)
        parity = np.array([[bin(a | b).count("1") & 1 for b in i] for a in i])
        return np.where(parity == 1, -1.0, 1.0)

    with pytest.raises(AssertionError):
        check_hadamard_matches_scipy(_Mutant(hadamard_matrix=bad_hadamard), 8)


def test_mutant_truncating_fp16_scale_is_caught():
    def bad_round(v):
        v = np.asarray(v, dtype=np.float64)
        h = np.clip(v, -O.FP16_MAX, O.FP16_MAX).astype(np.float16)
        up = h.astype(np.float64) > v  # round toward zero instead of to nearest
        h = np.where(up, np.nextafter(h, np.float16(0)), h)
        return h.astype(np.float64)

    with pytest.raises(AssertionError):
        check_fp16_scale_rounding(_Mutant(fp16_round=bad_round))


def test_mutant_floor_e8m0_exponent_is_caught():
    def bad_exp(v):
        v = np.asarray(v, dtype=np.float64)
        return np.clip(np.floor(np.log2(np.where(v > 0, v, 1.0))), -126, 127).astype(np.int64)

    def bad_store(a, fmt):
        e = bad_exp(a)
        return np.ldexp(1.0, e), (e + 127).astype(np.uint8)

    with pytest.raises(AssertionError):
        check_e8m0_scale(_Mutant(e8m0_exponent=bad_exp, store_scales=bad_store))
