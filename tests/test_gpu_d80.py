"""GPU parity at the head dimension d = 80 against the fp64 oracle, through
the C ABI.

d = 80 is the smallest size the survey of the pages names beside 96 and
192 for the SRFT's freedom from powers of two.  The SRFT is the packed
unitary DFT of length 80 (the oracle's general even-d form); the library runs
the codec as the tensor-core contraction padded to the 128-wide tile (R zero
outside its 80 x 80 block) and the bare transform as a dense map.  The code
rows are 40 (int4) or 80 (int8) bytes and a fp32 scale row is 20 bytes: not
rows a TMA tensor map can stride over, so the quantize stores them with
narrow stores and the dequantize reads them with plain bulk copies.  Groups
of 16 only (32 does not divide 80).  Sizes span several 128-row tiles with
ragged tails, windows inside a larger cache, both sides of one launch in
different widths.
"""

import numpy as np
import pytest
import torch

from oracle import srft_oracle as O
from int8_kv_cache_srft_gb300 import inputs as I
from tests.parity import assert_codes, assert_dequant_within_step, assert_reconstruction_bound, assert_scales
from tests.test_gpu_scale_formats import check_side as check_side_fmt

pytestmark = pytest.mark.gpu

K = None
D = 80


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global K
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import int8_kv_cache_srft_gb300 as mod

    mod.library()
    K = mod
    yield
    assert K.srftkv_device_fault() == 0


def _np(t):
    return t.detach().cpu().numpy()


def tm(t):
    return t.permute(0, 2, 1, 3)


@pytest.mark.parametrize("inverse", (False, True))
def test_transform_d80(inverse):
    g = torch.Generator().manual_seed(80)
    n = 1001
    x = (torch.randn((n, D), generator=g) * 3).to(torch.float16)
    y = torch.empty((n, D), dtype=torch.float32, device="cuda")
    K.srft_transform(x.cuda(), y, n, D, 7, inverse)
    torch.cuda.synchronize()
    xd = _np(x).astype(np.float64)
    ref = O.srft_inverse(xd, 7) if inverse else O.srft_forward(xd, 7)
    err = np.abs(_np(y) - ref).max(axis=-1)
    assert np.all(err <= 2e-6 * np.linalg.norm(xd, axis=-1) + 1e-7)


@pytest.mark.parametrize("bits,lam", [(b, l) for b in (4, 8) for l in (False, True)])
def test_codec_d80_ragged(bits, lam):
    """2 outer x 300 tokens x 3 heads (three 128-row tiles a head, the last ragged), written at t_offset 16 of
    t_cap 320; K and V of one launch in different widths; rows outside the window untouched."""
    n, T, H, t_cap, t_off, seed, group = 2, 300, 3, 320, 16, 11, 16
    w = I.Workload("d80", n_outer=n, tokens=T, kv_heads=H, d=D, lam=lam, data_seed=bits + 80,
                   outlier_kind="scale", outlier_channels=2, outlier_factor=30.0)
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    lk, lv = I.lam_table(w, "k"), I.lam_table(w, "v")
    bits_v = 12 - bits
    sides = []
    for x, l, b in ((xk, lk, bits), (xv, lv, bits_v)):
        s = K.alloc_side(n, t_cap, H, D, b, group)
        s.codes.fill_(0xAB)
        s.scales.fill_(-1.0)
        s.x = x.cuda()
        s.lam = None if l is None else l.cuda()
        sides.append(s)
    K.srft_kv_quantize(sides[0], sides[1], n, T, H, D, group, t_cap, t_off, seed)
    torch.cuda.synchronize()
    for s, x, l, b in ((sides[0], xk, lk, bits), (sides[1], xv, lv, bits_v)):
        lam_b = None if l is None else _np(l)[:, None, :, :]
        enc = O.srft_kv_quantize(_np(x).astype(np.float64), lam_b, b, group, seed)
        codes = _np(tm(s.codes))
        assert (codes[:, :t_off] == 0xAB).all() and (codes[:, t_off + T:] == 0xAB).all(), "rows outside the window"
        sc = _np(tm(s.scales))
        assert (sc[:, :t_off] == -1.0).all() and (sc[:, t_off + T:] == -1.0).all(), "scale rows outside the window"
        assert_scales(sc[:, t_off:t_off + T], enc["scales"])
        assert_codes(codes[:, t_off:t_off + T], enc["r"], b)
        out = torch.full_like(s.x, float("nan"))
        K.srft_kv_dequantize(K.Side(s.codes, s.scales, b, x=out, lam=s.lam), None, n, T, H, D, group, t_cap, t_off,
                             seed)
        torch.cuda.synchronize()
        xg = _np(out).astype(np.float64)
        assert np.isfinite(xg).all()
        lam_full = None if lam_b is None else np.broadcast_to(lam_b, x.shape)
        ref_hat = O.srft_kv_dequantize(enc["codes"], enc["scales"], lam_b, b, group, seed)
        assert_dequant_within_step(xg, ref_hat, enc["scales"], lam_full, group)
        assert_reconstruction_bound(xg, _np(x), enc["scales"], lam_full, group)
        mine = O.srft_kv_dequantize(codes[:, t_off:t_off + T], sc[:, t_off:t_off + T].astype(np.float64), lam_b, b,
                                    group, seed)
        assert np.abs(xg - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5


@pytest.mark.parametrize("fmt", ("fp16", "e8m0"))
@pytest.mark.parametrize("bits", (4, 8))
def test_codec_d80_scale_formats(fmt, bits):
    n, T, H, seed, group = 2, 320, 3, 19, 16
    w = I.Workload("d80sf", n_outer=n, tokens=T, kv_heads=H, d=D, lam=(bits == 4), data_seed=3 * bits + 80,
                   outlier_kind="scale", outlier_channels=2, outlier_factor=30.0)
    x, lam = I.kv_side(w, "k"), I.lam_table(w, "k")
    s = K.alloc_side(n, T, H, D, bits, group, scale_format=fmt)
    s.x = x.cuda()
    s.lam = None if lam is None else lam.cuda()
    K.srft_kv_quantize(s, None, n, T, H, D, group, T, 0, seed)
    torch.cuda.synchronize()
    enc, lam_b, raw = check_side_fmt(s, x, lam, bits, group, seed, fmt)
    out = torch.empty_like(s.x)
    K.srft_kv_dequantize(K.Side(s.codes, s.scales, bits, x=out, lam=s.lam, scale_format=fmt), None, n, T, H, D, group,
                         T, 0, seed)
    torch.cuda.synchronize()
    mine = O.srft_kv_dequantize(_np(tm(s.codes)), O.decode_scales(raw, fmt), lam_b, bits, group, seed)
    assert np.abs(_np(out) - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5


def test_codec_d80_small_call():
    """One token of one head (a partial tile, the append shape) takes the tensor-core path and matches."""
    n, T, H, seed = 1, 1, 1, 3
    w = I.Workload("d80small", n_outer=n, tokens=T, kv_heads=H, d=D, data_seed=5)
    x = I.kv_side(w, "k")
    s = K.alloc_side(n, 16, H, D, 4, 16)
    s.codes.fill_(0xAB)
    s.x = x.cuda()
    K.srft_kv_quantize(s, None, n, T, H, D, 16, 16, 7, seed)
    torch.cuda.synchronize()
    enc = O.srft_kv_quantize(_np(x).astype(np.float64), None, 4, 16, seed)
    assert_scales(_np(tm(s.scales))[:, 7:8], enc["scales"])
    assert_codes(_np(tm(s.codes))[:, 7:8], enc["r"], 4)
    codes = _np(tm(s.codes))
    assert (codes[:, :7] == 0xAB).all() and (codes[:, 8:] == 0xAB).all()


def test_dequant_d80_rows_not_on_16_bytes_rejected():
    """int4 code rows of 40 bytes: a window that starts on an odd token (t_offset 3: 120 bytes, not a multiple
    of 16) cannot be bulk-copied and is rejected before any launch."""
    s = K.alloc_side(1, 64, 1, D, 4, 16)
    out = torch.empty((1, 8, 1, D), dtype=torch.float16, device="cuda")
    with pytest.raises(RuntimeError, match="multiples of 16"):
        K.srft_kv_dequantize(K.Side(s.codes, s.scales, 4, x=out), None, 1, 8, 1, D, 16, 64, 3, 1)


def test_d80_decode_shape_sampled():
    """The decode cache shape at d = 80 cut to 4 sequences (4 x 131072 tokens x 8 kv heads = 4.2 M vectors a
    side), quantised and dequantised in one launch each: every scale row written, sampled rows against the
    oracle."""
    w = I.DECODE.resized(n_outer=4, d=D)
    B, Hkv, T, seed = w.n_outer, w.kv_heads, w.tokens, w.sign_seed
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    sk, sv = K.alloc_side(B, T, Hkv, D, 4, 16), K.alloc_side(B, T, Hkv, D, 4, 16)
    sk.x, sv.x = xk, xv
    K.srft_kv_quantize(sk, sv, B, T, Hkv, D, 16, T, 0, seed)
    ok_, ov_ = torch.empty_like(xk), torch.empty_like(xv)
    K.srft_kv_dequantize(K.Side(sk.codes, sk.scales, 4, x=ok_), K.Side(sv.codes, sv.scales, 4, x=ov_), B, T, Hkv, D,
                         16, T, 0, seed)
    torch.cuda.synchronize()
    gen = np.random.default_rng(80)
    for side, x, xhat in ((sk, xk, ok_), (sv, xv, ov_)):
        assert bool((side.scales > 0).all()), "unwritten scale rows"
        b, t, h = gen.integers(0, B, 2000), gen.integers(0, T, 2000), gen.integers(0, Hkv, 2000)
        bi, ti, hi = (torch.from_numpy(a).cuda() for a in (b, t, h))
        xs = _np(x[bi, ti, hi]).astype(np.float64)[:, None, :]
        enc = O.srft_kv_quantize(xs, None, 4, 16, seed)
        codes = _np(side.codes[bi, hi, ti])[:, None, :]
        scales = _np(side.scales[bi, hi, ti])[:, None, :]
        assert_scales(scales, enc["scales"])
        assert_codes(codes, enc["r"], 4)
        got = _np(xhat[bi, ti, hi]).astype(np.float64)[:, None, :]
        mine = O.srft_kv_dequantize(codes, scales.astype(np.float64), None, 4, 16, seed)
        assert np.abs(got - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5
