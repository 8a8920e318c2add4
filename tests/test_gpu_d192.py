"""GPU parity at d = 192 (a head dimension that is not a power of two, run as
a mixed-radix register transform, two lanes per vector) against the fp64
oracle, through the C ABI.

At d = 192 the SRFT is the packed unitary DFT of length 192 (the oracle's
general even-d form); the codec takes 96-point complex transforms split
across a lane pair (one radix-2 step, then 3 x 16 points in each lane), the
bare transform a dense map, and attention the dense q preparation and
combine of a non-power-of-two d.  Sizes span many 16-row tiles with ragged
tails and a window inside a larger cache, on both sides of one launch with
mixed widths.
"""

import numpy as np
import pytest
import torch

from oracle import srft_oracle as O
from int8_kv_cache_srft_gb300 import inputs as I
from tests.parity import ATTN_ATOL, assert_codes, assert_dequant_within_step, assert_reconstruction_bound, assert_scales
from tests.test_gpu_scale_formats import check_side as check_side_fmt
from tests.test_gpu_scale_formats import raw_np

pytestmark = pytest.mark.gpu

K = None
D = 192


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
def test_transform_d192(inverse):
    g = torch.Generator().manual_seed(192)
    n = 1001  # ragged: not a multiple of the four rows a block takes
    x = (torch.randn((n, D), generator=g) * 3).to(torch.float16)
    y = torch.empty((n, D), dtype=torch.float32, device="cuda")
    K.srft_transform(x.cuda(), y, n, D, 7, inverse)
    torch.cuda.synchronize()
    xd = _np(x).astype(np.float64)
    ref = O.srft_inverse(xd, 7) if inverse else O.srft_forward(xd, 7)
    err = np.abs(_np(y) - ref).max(axis=-1)
    assert np.all(err <= 2e-6 * np.linalg.norm(xd, axis=-1) + 1e-7)


@pytest.mark.parametrize("bits,group,lam", [(b, g, l) for b in (4, 8) for g in (16, 32, 64) for l in (False, True)])
def test_codec_d192_ragged(bits, group, lam):
    """2 outer x 300 tokens x 3 heads (19 tiles of 16 rows a head, the last one ragged), written at t_offset 16
    of t_cap 320; K and V of one launch in different widths; then the GPU decode of the GPU codes against the
    oracle's decode of the same codes."""
    n, T, H, t_cap, t_off, seed = 2, 300, 3, 320, 16, 11
    w = I.Workload("d192", n_outer=n, tokens=T, kv_heads=H, d=D, lam=lam, data_seed=bits + group,
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
        assert_scales(_np(tm(s.scales))[:, t_off:t_off + T], enc["scales"])
        assert_codes(codes[:, t_off:t_off + T], enc["r"], b)
        out = torch.empty_like(s.x)
        K.srft_kv_dequantize(K.Side(s.codes, s.scales, b, x=out, lam=s.lam), None, n, T, H, D, group, t_cap, t_off,
                             seed)
        torch.cuda.synchronize()
        xg = _np(out).astype(np.float64)
        lam_full = None if lam_b is None else np.broadcast_to(lam_b, x.shape)
        ref_hat = O.srft_kv_dequantize(enc["codes"], enc["scales"], lam_b, b, group, seed)
        assert_dequant_within_step(xg, ref_hat, enc["scales"], lam_full, group)
        assert_reconstruction_bound(xg, _np(x), enc["scales"], lam_full, group)
        mine = O.srft_kv_dequantize(codes[:, t_off:t_off + T], _np(tm(s.scales))[:, t_off:t_off + T].astype(np.float64),
                                    lam_b, b, group, seed)
        assert np.abs(xg - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5


@pytest.mark.parametrize("fmt", ("fp16", "e8m0"))
@pytest.mark.parametrize("bits,group", ((4, 16), (4, 32), (8, 16), (4, 64)))
def test_codec_d192_scale_formats(fmt, bits, group):
    n, T, H, seed = 2, 321, 3, 19
    w = I.Workload("d192sf", n_outer=n, tokens=T, kv_heads=H, d=D, lam=(bits == 4), data_seed=3 * bits + group,
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


def test_codec_d192_single_token_and_zero_rows():
    """A one-token append (one partial tile, 15 of its 16 rows past the end) and all-zero rows."""
    n, H, seed = 2, 3, 3
    w = I.Workload("d192one", n_outer=n, tokens=1, kv_heads=H, d=D, data_seed=5)
    x = I.kv_side(w, "k")
    x[1] = 0
    s = K.alloc_side(n, 8, H, D, 4, 16)
    s.codes.fill_(0xAB)
    s.x = x.cuda()
    K.srft_kv_quantize(s, None, n, 1, H, D, 16, 8, 5, seed)
    torch.cuda.synchronize()
    enc = O.srft_kv_quantize(_np(x).astype(np.float64), None, 4, 16, seed)
    assert_scales(_np(tm(s.scales))[:, 5:6], enc["scales"])
    assert_codes(_np(tm(s.codes))[:, 5:6], enc["r"], 4)
    codes = _np(tm(s.codes))
    assert (codes[:, :5] == 0xAB).all() and (codes[:, 6:] == 0xAB).all()
    assert not codes[1, 5].any() and not _np(tm(s.scales))[1, 5].any()


# ---------------------------------------------------------------------------
# decode attention at d = 192
# ---------------------------------------------------------------------------
from tests.test_gpu_attention import build_cache, oracle_attention, run_attention  # noqa: E402

ATTN192 = [(bk, bv, g) for bk, bv in ((4, 4), (8, 4), (4, 8), (8, 8), (16, 16)) for g in (16, 32)
           if bk != 16 or g == 16]  # the raw fp16 cache has no groups


@pytest.fixture()
def attn_helpers():
    """The attention tests' cache builder, bound to this module's library handle."""
    import tests.test_gpu_attention as TA

    TA.K = K
    return TA


@pytest.mark.parametrize("bk,bv,group", ATTN192)
def test_attention_d192_matches_oracle(attn_helpers, bk, bv, group):
    """Ragged lengths (300 and 137) over t_cap 300, four query heads per kv head, lambda on."""
    B, Hkv, rep, t_cap, seed = 2, 2, 4, 300, 21
    Hq = Hkv * rep
    sk, sv = build_cache(B, Hkv, D, t_cap, bk, bv, group, seed, lam=(bk != 16), data_seed=bk * 10 + bv + group)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=D, q_heads=Hq, data_seed=192), device="cuda")
    seq = torch.tensor([300, 137], dtype=torch.int32, device="cuda")
    out = run_attention(q, sk, sv, B, Hq, Hkv, D, group, t_cap, seq, seed)
    ref = oracle_attention(q, sk, sv, group, seed, seq)
    err = np.abs(out - ref).max()
    assert err <= ATTN_ATOL, f"max-abs error {err:.3g}"


@pytest.mark.parametrize("rep,n_splits", ((1, 0), (2, 1), (3, 5), (4, 0)))
def test_attention_d192_gqa_and_splits(attn_helpers, rep, n_splits):
    B, Hkv, t_cap, seed = 3, 2, 1000, 8
    Hq = Hkv * rep
    sk, sv = build_cache(B, Hkv, D, t_cap, 4, 4, 16, seed, data_seed=rep)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=D, q_heads=Hq, data_seed=rep + 50), device="cuda")
    seq = torch.tensor([1000, 1, 517], dtype=torch.int32, device="cuda")
    out = run_attention(q, sk, sv, B, Hq, Hkv, D, 16, t_cap, seq, seed, n_splits=n_splits, sm_scale=0.11)
    ref = oracle_attention(q, sk, sv, 16, seed, seq, sm_scale=0.11)
    assert np.abs(out - ref).max() <= ATTN_ATOL


@pytest.mark.parametrize("fmt_k,fmt_v,group", (("fp16", "fp16", 16), ("e8m0", "e8m0", 16), ("fp32", "e8m0", 32),
                                               ("fp16", "fp32", 32)))
def test_attention_d192_scale_formats(fmt_k, fmt_v, group):
    B, Hkv, rep, t_cap, seed = 2, 2, 4, 320, 31
    w = I.Workload("attn192", n_outer=B, tokens=t_cap, kv_heads=Hkv, d=D, lam=True, data_seed=group,
                   outlier_kind="scale", outlier_channels=2, outlier_factor=8.0)
    sides = []
    for name, fmt in (("k", fmt_k), ("v", fmt_v)):
        x, lam = I.kv_side(w, name), I.lam_table(w, name)
        s = K.alloc_side(B, t_cap, Hkv, D, 4, group, scale_format=fmt)
        s.x, s.lam = x.cuda(), lam.cuda()
        K.srft_kv_quantize(s, None, B, t_cap, Hkv, D, group, t_cap, 0, seed)
        sides.append(s)
    torch.cuda.synchronize()
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=D, q_heads=Hkv * rep, data_seed=7), device="cuda")
    seq = torch.tensor([320, 97], dtype=torch.int32, device="cuda")
    out = torch.empty((B, Hkv * rep, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hkv * rep, Hkv, D, t_cap, 0), dtype=torch.uint8,
                     device="cuda")
    K.q4kv_decode_attention(q, out, sides[0], sides[1], B, Hkv * rep, Hkv, D, group, t_cap, seq, 0.0, seed, 0, ws)
    torch.cuda.synchronize()

    def oside(s, fmt):
        return {"bits": 4, "codes": _np(tm(s.codes)), "scales": O.decode_scales(raw_np(s.scales, fmt), fmt),
                "lam": _np(s.lam).astype(np.float64), "group": group}

    ref = O.packed_decode_attention(_np(q).astype(np.float64), oside(sides[0], fmt_k), oside(sides[1], fmt_v), seed,
                                    _np(seq))
    assert np.abs(_np(out) - ref).max() <= ATTN_ATOL


def test_d192_decode_shape_full_size_sampled():
    """The decode workload's cache shape at d = 192 (B=16, Hkv=8, T=131072, Hq=32; the bench's d = 192
    variant, in the launch configuration it times): the whole cache quantised and dequantised in one launch
    each, attention over all of it with the automatic split count; rows and (b, kv head) pairs sampled for the
    oracle."""
    w = I.DECODE.resized(d=D)
    B, Hkv, T, Hq, seed = w.n_outer, w.kv_heads, w.tokens, w.q_heads, w.sign_seed
    rep = Hq // Hkv
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    sk, sv = K.alloc_side(B, T, Hkv, D, 4, 16), K.alloc_side(B, T, Hkv, D, 4, 16)
    sk.x, sv.x = xk, xv
    K.srft_kv_quantize(sk, sv, B, T, Hkv, D, 16, T, 0, seed)
    ok_, ov_ = torch.empty_like(xk), torch.empty_like(xv)
    K.srft_kv_dequantize(K.Side(sk.codes, sk.scales, 4, x=ok_), K.Side(sv.codes, sv.scales, 4, x=ov_), B, T, Hkv, D,
                         16, T, 0, seed)
    q = I.query(w, device="cuda")
    out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, D, T, 0), dtype=torch.uint8, device="cuda")
    K.q4kv_decode_attention(q, out, sk, sv, B, Hq, Hkv, D, 16, T, None, 0.0, seed, 0, ws)
    torch.cuda.synchronize()
    out = _np(out)
    gen = np.random.default_rng(192)
    qn = _np(q).astype(np.float64)
    for b, h in ((0, 0), (B - 1, Hkv - 1), (7, 3)):
        rows = np.sort(gen.choice(T, 256, replace=False))
        for side, x, xhat in ((sk, xk, ok_), (sv, xv, ov_)):
            xs = _np(x[b, rows, h]).astype(np.float64)[None, :, None, :]
            enc = O.srft_kv_quantize(xs, None, 4, 16, seed)
            codes = _np(side.codes[b, h, rows])[None, :, None, :]
            scales = _np(side.scales[b, h, rows])[None, :, None, :]
            assert_scales(scales, enc["scales"])
            assert_codes(codes, enc["r"], 4)
            mine = O.srft_kv_dequantize(codes, scales.astype(np.float64), None, 4, 16, seed)
            got = _np(xhat[b, rows, h]).astype(np.float64)[None, :, None, :]
            assert np.abs(got - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5
        kh = O.srft_kv_dequantize(_np(sk.codes[b, h]), _np(sk.scales[b, h]).astype(np.float64), None, 4, 16, seed)
        vh = O.srft_kv_dequantize(_np(sv.codes[b, h]), _np(sv.scales[b, h]).astype(np.float64), None, 4, 16, seed)
        for r in range(rep):
            hq = h * rep + r
            s = kh @ qn[b, hq] / np.sqrt(D)
            pw = np.exp(s - s.max())
            ref = (pw @ vh) / pw.sum()
            assert np.abs(out[b, hq] - ref).max() <= ATTN_ATOL
