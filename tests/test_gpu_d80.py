"""GPU parity at the head dimension d = 80 against the fp64 oracle, through
the C ABI.

d = 80 is the smallest of the head sizes that are not powers of two (80, 96,
192) the library takes, sizes the SRFT covers where a Hadamard rotation
cannot ([WQF] Methodology 1).  The SRFT is the packed
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


# ---------------------------------------------------------------------------
# decode attention at d = 80 (int4 rows of 40 bytes are read as rows of token pairs)
# ---------------------------------------------------------------------------
from tests.test_gpu_attention import build_cache, oracle_attention, run_attention  # noqa: E402
from tests.test_gpu_scale_formats import raw_np  # noqa: E402
from tests.parity import ATTN_ATOL  # noqa: E402


@pytest.fixture()
def attn_helpers():
    """The attention tests' cache builder, bound to this module's library handle."""
    import tests.test_gpu_attention as TA

    TA.K = K
    return TA


@pytest.mark.parametrize("bk,bv", ((4, 4), (8, 4), (4, 8), (8, 8), (16, 16)))
def test_attention_d80_matches_oracle(attn_helpers, bk, bv):
    """Ragged lengths (300 = 9 chunks + 12, and 137: a pair row with only its even token) over t_cap 300, four
    query heads per kv head, lambda on; both pair-row sides, both mixed ones and the raw fp16 cache."""
    B, Hkv, rep, t_cap, seed = 2, 2, 4, 300, 21
    Hq = Hkv * rep
    sk, sv = build_cache(B, Hkv, D, t_cap, bk, bv, 16, seed, lam=(bk != 16), data_seed=bk * 10 + bv + 80)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=D, q_heads=Hq, data_seed=80), device="cuda")
    seq = torch.tensor([300, 137], dtype=torch.int32, device="cuda")
    out = run_attention(q, sk, sv, B, Hq, Hkv, D, 16, t_cap, seq, seed)
    ref = oracle_attention(q, sk, sv, 16, seed, seq)
    err = np.abs(out - ref).max()
    assert err <= ATTN_ATOL, f"max-abs error {err:.3g}"


@pytest.mark.parametrize("rep,n_splits,bk,bv", ((1, 0, 4, 4), (2, 1, 4, 4), (3, 5, 8, 4), (6, 0, 4, 4),
                                                (4, 3, 4, 8)))
def test_attention_d80_gqa_and_splits(attn_helpers, rep, n_splits, bk, bv):
    """GQA 1, 2, 3, 6 (two head groups) and split counts from one to automatic; sequence lengths 1000, 1, 517."""
    B, Hkv, t_cap, seed = 3, 2, 1000, 8
    Hq = Hkv * rep
    sk, sv = build_cache(B, Hkv, D, t_cap, bk, bv, 16, seed, data_seed=rep + 80)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=D, q_heads=Hq, data_seed=rep + 50), device="cuda")
    seq = torch.tensor([1000, 1, 517], dtype=torch.int32, device="cuda")
    out = run_attention(q, sk, sv, B, Hq, Hkv, D, 16, t_cap, seq, seed, n_splits=n_splits, sm_scale=0.11)
    ref = oracle_attention(q, sk, sv, 16, seed, seq, sm_scale=0.11)
    assert np.abs(out - ref).max() <= ATTN_ATOL


@pytest.mark.parametrize("fmt_k,fmt_v", (("fp16", "fp16"), ("e8m0", "e8m0"), ("fp32", "e8m0"), ("fp16", "fp32")))
def test_attention_d80_scale_formats(fmt_k, fmt_v):
    B, Hkv, rep, t_cap, seed, group = 2, 2, 4, 320, 31, 16
    w = I.Workload("attn80", n_outer=B, tokens=t_cap, kv_heads=Hkv, d=D, lam=True, data_seed=80,
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


def test_attention_d80_v_scales_far_from_one(attn_helpers):
    """V scales times 2^-18 and 2^12 (exact powers of two: the warp reruns its chunks with a V unit) on pair
    rows: the output is that of the unscaled cache times the same factor."""
    B, Hkv, rep, t_cap, seed = 1, 2, 4, 256, 5
    Hq = Hkv * rep
    sk, sv = build_cache(B, Hkv, D, t_cap, 4, 4, 16, seed, data_seed=81)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=D, q_heads=Hq, data_seed=82), device="cuda")
    o1 = run_attention(q, sk, sv, B, Hq, Hkv, D, 16, t_cap, None, seed)
    ref = oracle_attention(q, sk, sv, 16, seed, None)
    assert np.abs(o1 - ref).max() <= ATTN_ATOL
    base = sv.scales.clone()
    for f in (2.0**-18, 2.0**12):
        sv.scales.copy_(base * f)
        of = run_attention(q, sk, sv, B, Hq, Hkv, D, 16, t_cap, None, seed)
        assert np.isfinite(of).all()
        assert np.abs(of / f - o1).max() <= 1e-5 * max(1.0, float(np.abs(o1).max()))


def test_attention_d80_rejects_misaligned_t_cap():
    """fp32 group-16 rows are 20 bytes at d = 80: a t_cap that leaves a (batch, kv head)'s scales off the 16-byte
    rows the copy uses (or an odd one, which splits a token pair) is rejected."""
    B, Hkv = 1, 1
    for t_cap in (33, 34):
        sk = K.alloc_side(B, t_cap, Hkv, D, 4, 16)
        sv = K.alloc_side(B, t_cap, Hkv, D, 4, 16)
        q = torch.zeros((B, 4, D), dtype=torch.float16, device="cuda")
        out = torch.empty((B, 4, D), dtype=torch.float32, device="cuda")
        ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, 4, Hkv, D, t_cap, 0), dtype=torch.uint8,
                         device="cuda")
        with pytest.raises(RuntimeError, match="multiple of 16|even t_cap"):
            K.q4kv_decode_attention(q, out, sk, sv, B, 4, Hkv, D, 16, t_cap, None, 0.0, 1, 0, ws)


def test_d80_decode_shape_full_size_sampled():
    """The decode workload's cache shape at d = 80 (B=16, Hkv=8, T=131072, Hq=32; the bench's d = 80 variant, in
    the launch configuration it times): the whole cache quantised and dequantised in one launch each, attention
    over all of it with the automatic split count; every scale row written, rows and (b, kv head) pairs sampled
    for the oracle."""
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
    assert bool((sk.scales > 0).all()) and bool((sv.scales > 0).all()), "unwritten scale rows"
    gen = np.random.default_rng(80)
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
