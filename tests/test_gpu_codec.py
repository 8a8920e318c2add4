"""GPU parity of the codec kernels (quantize, dequantize, bare transform)
against the fp64 oracle, through the C ABI.

Sizes: the full tiny workload, reduced versions of the Gemma-, Qwen- and
K8V4-shaped workloads that span many 32-row tiles with ragged tails, and the
full-size Qwen-shaped and K8V4 caches in the launch configuration the
benchmark uses, checked on seeded samples of rows.
"""

import numpy as np
import pytest
import torch

from oracle import srft_oracle as O
from int8_kv_cache_srft_gb300 import inputs as I
from tests.parity import assert_codes, assert_dequant_within_step, assert_reconstruction_bound, assert_scales

pytestmark = pytest.mark.gpu

K = None


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
    """Token-major view [outer][token][head][...] of a head-major plane [outer][head][token][...]."""
    return t.permute(0, 2, 1, 3)


def hm_rows(rows, T, H):
    """Head-major row indices of token-major rows (o*T + t)*H + h of a [outer][T][H] array."""
    o, rem = rows // (T * H), rows % (T * H)
    return (o * H + rem % H) * T + rem // H


def _quantize_gpu(x_k, x_v, lam_k, lam_v, bits_k, bits_v, group, seed, t_cap=None, t_offset=0, sentinel=0xAB):
    n_outer, T, H, d = x_k.shape
    t_cap = T if t_cap is None else t_cap
    sk = K.alloc_side(n_outer, t_cap, H, d, bits_k, group)
    sv = K.alloc_side(n_outer, t_cap, H, d, bits_v, group)
    for s in (sk, sv):
        s.codes.fill_(sentinel)
        s.scales.fill_(-1.0)
    sk.x, sv.x = x_k.cuda(), x_v.cuda()
    sk.lam = None if lam_k is None else lam_k.cuda()
    sv.lam = None if lam_v is None else lam_v.cuda()
    K.srft_kv_quantize(sk, sv, n_outer, T, H, d, group, t_cap, t_offset, seed)
    torch.cuda.synchronize()
    return sk, sv


def _oracle(x, lam, bits, group, seed):
    lam_b = None if lam is None else _np(lam)[:, None, :, :]
    return O.srft_kv_quantize(_np(x).astype(np.float64), lam_b, bits, group, seed), lam_b


def _check_side(side, x, lam, bits, group, seed, t_offset=0):
    T = x.shape[1]
    enc, lam_b = _oracle(x, lam, bits, group, seed)
    codes = _np(tm(side.codes))[:, t_offset : t_offset + T]
    scales = _np(tm(side.scales))[:, t_offset : t_offset + T]
    assert_scales(scales, enc["scales"])
    st = assert_codes(codes, enc["r"], bits)
    return enc, lam_b, st


@pytest.mark.parametrize("d", (16, 32, 64, 128, 256))
@pytest.mark.parametrize("inverse", (False, True))
def test_transform_matches_oracle(d, inverse):
    g = torch.Generator().manual_seed(d)
    n = 1000  # ragged: not a multiple of the 128-thread block
    x = (torch.randn((n, d), generator=g) * 3).to(torch.float16)
    y = torch.empty((n, d), dtype=torch.float32, device="cuda")
    K.srft_transform(x.cuda(), y, n, d, 7, inverse)
    torch.cuda.synchronize()
    xd = _np(x).astype(np.float64)
    ref = O.srft_inverse(xd, 7) if inverse else O.srft_forward(xd, 7)
    err = np.abs(_np(y) - ref).max(axis=-1)
    assert np.all(err <= 2e-6 * np.linalg.norm(xd, axis=-1) + 1e-7)


def test_tiny_round_trip_workload():
    w = I.TINY
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    sk, sv = _quantize_gpu(xk, xv, None, None, 4, 4, w.group, w.sign_seed)
    for side, x in ((sk, xk), (sv, xv)):
        enc, _, _ = _check_side(side, x, None, 4, w.group, w.sign_seed)
        out = torch.empty_like(side.x)
        dq = K.Side(side.codes, side.scales, 4, x=out)
        K.srft_kv_dequantize(dq, None, 1, w.tokens, w.kv_heads, w.d, w.group, w.tokens, 0, w.sign_seed)
        torch.cuda.synchronize()
        xg = _np(out).astype(np.float64)
        ref_hat = O.srft_kv_dequantize(enc["codes"], enc["scales"], None, 4, w.group, w.sign_seed)
        assert_dequant_within_step(xg, ref_hat, enc["scales"], None, w.group)
        assert_reconstruction_bound(xg, _np(x), enc["scales"], None, w.group)
        # tight: the GPU decode of the GPU codes against the oracle decode of the same codes
        ref = O.srft_kv_dequantize(_np(tm(side.codes)), _np(tm(side.scales)).astype(np.float64), None, 4, w.group,
                                   w.sign_seed)
        assert np.abs(xg - ref).max() <= np.abs(ref).max() * 2.0**-10 + 1e-5


CASES = [(d, bits, group, lam) for d in (16, 32, 64, 128, 256) for bits in (4, 8)
         for group in sorted({16, d}) for lam in (False, True)]


@pytest.mark.parametrize("d,bits,group,lam", CASES)
def test_quantize_dequantize_ragged(d, bits, group, lam):
    """2 outer x 37 tokens x 3 heads = 111 rows per outer (ragged tiles), written at t_offset 5 of t_cap 50."""
    w = I.Workload("ragged", n_outer=2, tokens=37, kv_heads=3, d=d, lam=lam, data_seed=d + bits,
                   outlier_kind="scale", outlier_channels=2, outlier_factor=30.0)
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    lk, lv = I.lam_table(w, "k"), I.lam_table(w, "v")
    bits_v = 12 - bits  # the other width on the V side: exercises one launch with mixed widths
    sk, sv = _quantize_gpu(xk, xv, lk, lv, bits, bits_v, group, 11, t_cap=50, t_offset=5)
    for side, x, lam_t, b in ((sk, xk, lk, bits), (sv, xv, lv, bits_v)):
        enc, lam_b, _ = _check_side(side, x, lam_t, b, group, 11, t_offset=5)
        codes = _np(tm(side.codes))
        assert (codes[:, :5] == 0xAB).all() and (codes[:, 42:] == 0xAB).all(), "rows outside the window were written"
        out = torch.empty_like(side.x)
        dq = K.Side(side.codes, side.scales, b, x=out, lam=side.lam)
        K.srft_kv_dequantize(dq, None, 2, 37, 3, d, group, 50, 5, 11)
        torch.cuda.synchronize()
        lam_full = None if lam_b is None else np.broadcast_to(lam_b, x.shape)
        ref_hat = O.srft_kv_dequantize(enc["codes"], enc["scales"], lam_b, b, group, 11)
        assert_dequant_within_step(_np(out), ref_hat, enc["scales"], lam_full, group)
        assert_reconstruction_bound(_np(out), _np(x), enc["scales"], lam_full, group)


TC_CASES = [(bk, bv, group, lam) for bk, bv in ((4, 4), (8, 8), (8, 4), (4, 8)) for group in (16, 32, 64)
            for lam in (False, True)]


@pytest.mark.parametrize("bk,bv,group,lam", TC_CASES)
def test_tensor_core_quantize_path(monkeypatch, bk, bv, group, lam):
    """d = 128 through the tensor-core contraction (forced on for a small, ragged call): 3 outer x 300 tokens x
    3 heads = 900 rows per outer (7 tiles of 128 with a ragged last one), written at t_offset 3 of t_cap 310."""
    monkeypatch.setenv("SRFTKV_QUANT_PATH", "tc")
    w = I.Workload("tc", n_outer=3, tokens=300, kv_heads=3, d=128, lam=lam, data_seed=bk * 100 + bv * 10 + group,
                   outlier_kind="scale", outlier_channels=4, outlier_factor=50.0)
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    lk, lv = I.lam_table(w, "k"), I.lam_table(w, "v")
    sk, sv = _quantize_gpu(xk, xv, lk, lv, bk, bv, group, 13, t_cap=310, t_offset=3)
    for side, x, lam_t, b in ((sk, xk, lk, bk), (sv, xv, lv, bv)):
        enc, lam_b, _ = _check_side(side, x, lam_t, b, group, 13, t_offset=3)
        codes = _np(tm(side.codes))
        assert (codes[:, :3] == 0xAB).all() and (codes[:, 303:] == 0xAB).all()
        # and back through the tensor-core dequantize
        out = torch.empty_like(side.x)
        K.srft_kv_dequantize(K.Side(side.codes, side.scales, b, x=out, lam=side.lam), None, 3, 300, 3, 128, group,
                             310, 3, 13)
        torch.cuda.synchronize()
        lam_full = None if lam_b is None else np.broadcast_to(lam_b, x.shape)
        ref_hat = O.srft_kv_dequantize(enc["codes"], enc["scales"], lam_b, b, group, 13)
        assert_dequant_within_step(_np(out), ref_hat, enc["scales"], lam_full, group)
        assert_reconstruction_bound(_np(out), _np(x), enc["scales"], lam_full, group)
        mine = O.srft_kv_dequantize(codes[:, 3:303], _np(tm(side.scales))[:, 3:303].astype(np.float64), lam_b, b, group,
                                    13)
        assert np.abs(_np(out) - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5


def test_lambda_fold_mixed_sides_and_broadcast(monkeypatch):
    """The tensor-core dequantize folds 1/lambda into its B operand and rebuilds it whenever the lambda row of
    its tiles changes.  K with one lambda table broadcast over the outer index (outer stride 0) and V without
    lambda go through one launch; 3 outer x 1100 tokens x 4 heads (9 tiles of 128 a head, 216 tiles) so the
    contiguous tile range of a CTA straddles heads and the K/V boundary."""
    monkeypatch.setenv("SRFTKV_QUANT_PATH", "tc")
    n, T, H, d, g, seed = 3, 1100, 4, 128, 16, 29
    w = I.Workload("fold", n_outer=n, tokens=T, kv_heads=H, d=d, lam=True, data_seed=29,
                   outlier_kind="scale", outlier_channels=4, outlier_factor=50.0)
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    lk = I.lam_table(w, "k", n_outer=1)  # [1][H][d]: one table for every outer index
    sk, sv = _quantize_gpu(xk, xv, lk, None, 4, 4, g, seed)
    enc_k, lam_b, _ = _check_side(sk, xk, lk, 4, g, seed)
    enc_v, _, _ = _check_side(sv, xv, None, 4, g, seed)
    outk, outv = torch.empty_like(sk.x), torch.empty_like(sv.x)
    K.srft_kv_dequantize(K.Side(sk.codes, sk.scales, 4, x=outk, lam=sk.lam), K.Side(sv.codes, sv.scales, 4, x=outv),
                         n, T, H, d, g, T, 0, seed)
    torch.cuda.synchronize()
    for side, out, lam_side in ((sk, outk, lam_b), (sv, outv, None)):
        mine = O.srft_kv_dequantize(_np(tm(side.codes)), _np(tm(side.scales)).astype(np.float64), lam_side, 4, g, seed)
        assert np.abs(_np(out) - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5


def test_zero_rows_and_empty_calls():
    x = torch.zeros((1, 40, 2, 128), dtype=torch.float16)
    sk, sv = _quantize_gpu(x, x, None, None, 4, 8, 16, 3)
    assert not _np(sk.scales).any() and not _np(sk.codes).any()
    assert not _np(sv.scales).any() and not _np(sv.codes).any()
    # n_tokens == 0 and n_outer == 0 are no-ops
    K.srft_kv_quantize(sk, sv, 1, 0, 2, 128, 16, 40, 0, 3)
    K.srft_kv_quantize(sk, sv, 0, 40, 2, 128, 16, 40, 0, 3)
    torch.cuda.synchronize()
    assert not _np(sk.codes).any()


def test_gemma_shaped_reduced():
    w = I.GEMMA
    xk, xv = I.kv_side(w, "k", n_outer=3, tokens=300), I.kv_side(w, "v", n_outer=3, tokens=300)
    sk, sv = _quantize_gpu(xk, xv, None, None, 4, 4, 16, w.sign_seed)
    for side, x in ((sk, xk), (sv, xv)):
        _check_side(side, x, None, 4, 16, w.sign_seed)


PAIR_CASES = [(group, bits, lam, tr) for group in (32, 64, 128) for bits in (4, 8) for lam in (False, True)
              for tr in ("srft", "srht")]


@pytest.mark.parametrize("group,bits,lam,tr", PAIR_CASES)
def test_d256_groups_between_16_and_d(group, bits, lam, tr):
    """d = 256 (two lanes per vector, each group's coordinates split between them) at the group sizes between
    16 and d: 2 outer x 75 tokens x 2 heads (16-row tiles with a ragged last one) at t_offset 3 of t_cap 80,
    the other width on V, then the GPU decode of the GPU codes against the oracle's decode of the same codes."""
    w = I.Workload("pair", n_outer=2, tokens=75, kv_heads=2, d=256, lam=lam, data_seed=group + bits,
                   outlier_kind="scale", outlier_channels=3, outlier_factor=40.0)
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    lk, lv = I.lam_table(w, "k"), I.lam_table(w, "v")
    bits_v = 12 - bits
    sides = []
    for x, lam_t, b in ((xk, lk, bits), (xv, lv, bits_v)):
        s = K.alloc_side(2, 80, 2, 256, b, group, transform=tr)
        s.codes.fill_(0xAB)
        s.scales.fill_(-1.0)
        s.x, s.lam = x.cuda(), None if lam_t is None else lam_t.cuda()
        sides.append(s)
    K.srft_kv_quantize(sides[0], sides[1], 2, 75, 2, 256, group, 80, 3, 19)
    torch.cuda.synchronize()
    for side, x, lam_t, b in ((sides[0], xk, lk, bits), (sides[1], xv, lv, bits_v)):
        lam_b = None if lam_t is None else _np(lam_t)[:, None, :, :]
        enc = O.srft_kv_quantize(_np(x).astype(np.float64), lam_b, b, group, 19, transform=tr)
        codes = _np(tm(side.codes))
        assert_scales(_np(tm(side.scales))[:, 3:78], enc["scales"])
        assert_codes(codes[:, 3:78], enc["r"], b)
        assert (codes[:, :3] == 0xAB).all() and (codes[:, 78:] == 0xAB).all(), "rows outside the window were written"
        out = torch.empty_like(side.x)
        K.srft_kv_dequantize(K.Side(side.codes, side.scales, b, x=out, lam=side.lam, transform=tr), None, 2, 75, 2,
                             256, group, 80, 3, 19)
        torch.cuda.synchronize()
        mine = O.srft_kv_dequantize(codes[:, 3:78], _np(tm(side.scales))[:, 3:78].astype(np.float64), lam_b, b, group,
                                    19, transform=tr)
        assert np.abs(_np(out) - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5


def test_gemma_shaped_full_size_sampled():
    """The full Gemma-3-1B-shaped cache (26 x 4096 x 1 x 256), K and V quantised in one launch and dequantised
    in one launch, as the benchmark times them; 2000 sampled rows per side against the oracle."""
    w = I.GEMMA
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    n_outer, T, H, d = xk.shape
    sk, sv = K.alloc_side(n_outer, T, H, d, 4, 16), K.alloc_side(n_outer, T, H, d, 4, 16)
    sk.x, sv.x = xk, xv
    K.srft_kv_quantize(sk, sv, n_outer, T, H, d, 16, T, 0, w.sign_seed)
    outk, outv = torch.empty_like(xk), torch.empty_like(xv)
    K.srft_kv_dequantize(K.Side(sk.codes, sk.scales, 4, x=outk), K.Side(sv.codes, sv.scales, 4, x=outv), n_outer, T, H,
                         d, 16, T, 0, w.sign_seed)
    torch.cuda.synchronize()
    rows = _sample_rows(n_outer * T * H, 2000, 47)
    hrows = torch.as_tensor(hm_rows(rows, T, H), device="cuda")
    for side, x, out in ((sk, xk, outk), (sv, xv, outv)):
        xs = _np(x.reshape(-1, d)[rows]).astype(np.float64)
        enc = O.srft_kv_quantize(xs, None, 4, 16, w.sign_seed)
        assert_scales(_np(side.scales.reshape(-1, d // 16)[hrows]), enc["scales"])
        assert_codes(_np(side.codes.reshape(-1, d // 2)[hrows]), enc["r"], 4)
        xg = _np(out.reshape(-1, d)[rows]).astype(np.float64)
        ref_hat = O.srft_kv_dequantize(enc["codes"], enc["scales"], None, 4, 16, w.sign_seed)
        assert_dequant_within_step(xg, ref_hat, enc["scales"], None, 16)
        assert_reconstruction_bound(xg, xs, enc["scales"], None, 16)


def test_qwen_shaped_reduced_with_lambda():
    w = I.QWEN
    xk, xv = I.kv_side(w, "k", n_outer=2, tokens=700), I.kv_side(w, "v", n_outer=2, tokens=700)
    lk, lv = I.lam_table(w, "k", n_outer=2), I.lam_table(w, "v", n_outer=2)
    sk, sv = _quantize_gpu(xk, xv, lk, lv, 4, 4, 16, w.sign_seed)
    for side, x, lam in ((sk, xk, lk), (sv, xv, lv)):
        _check_side(side, x, lam, 4, 16, w.sign_seed)


def _sample_rows(n_rows, k, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.integers(0, n_rows, k), [0, n_rows - 1]]))


@pytest.mark.parametrize("path", ("tc", "fft"))
def test_qwen_shaped_full_size_sampled(monkeypatch, path):
    """The full 28 x 32768 x 2 x 128 cache with lambda, quantised in one launch; 3000 sampled rows per side
    against the oracle, then the dequantised rows within one step and the reconstruction MSE reported.  Both
    quantize paths (tensor-core contraction and register FFT) are checked."""
    monkeypatch.setenv("SRFTKV_QUANT_PATH", path)
    w = I.QWEN
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    lk, lv = I.lam_table(w, "k", device="cuda"), I.lam_table(w, "v", device="cuda")
    n_outer, T, H, d = xk.shape
    sk, sv = K.alloc_side(n_outer, T, H, d, 4, 16), K.alloc_side(n_outer, T, H, d, 4, 16)
    sk.x, sv.x, sk.lam, sv.lam = xk, xv, lk, lv
    K.srft_kv_quantize(sk, sv, n_outer, T, H, d, 16, T, 0, w.sign_seed)
    outk, outv = torch.empty_like(xk), torch.empty_like(xv)
    K.srft_kv_dequantize(K.Side(sk.codes, sk.scales, 4, x=outk, lam=lk), K.Side(sv.codes, sv.scales, 4, x=outv, lam=lv),
                         n_outer, T, H, d, 16, T, 0, w.sign_seed)
    torch.cuda.synchronize()
    rows = _sample_rows(n_outer * T * H, 3000, 33)
    for side, x, lam, out in ((sk, xk, lk, outk), (sv, xv, lv, outv)):
        xs = _np(x.reshape(-1, d)[rows]).astype(np.float64)
        o_idx, h_idx = rows // (T * H), rows % H
        lam_rows = _np(lam)[o_idx, h_idx]
        enc = O.srft_kv_quantize(xs, lam_rows, 4, 16, w.sign_seed)
        hrows = torch.as_tensor(hm_rows(rows, T, H), device="cuda")
        assert_scales(_np(side.scales.reshape(-1, d // 16)[hrows]), enc["scales"])
        assert_codes(_np(side.codes.reshape(-1, d // 2)[hrows]), enc["r"], 4)
        xg = _np(out.reshape(-1, d)[rows]).astype(np.float64)
        ref_hat = O.srft_kv_dequantize(enc["codes"], enc["scales"], lam_rows, 4, 16, w.sign_seed)
        assert_dequant_within_step(xg, ref_hat, enc["scales"], lam_rows, 16)
        assert_reconstruction_bound(xg, xs, enc["scales"], lam_rows, 16)
        # reconstruction MSE of the GPU path and of the oracle agree closely
        mse_gpu, mse_ref = float(((xg - xs) ** 2).mean()), float(((ref_hat - xs) ** 2).mean())
        assert abs(mse_gpu - mse_ref) <= 0.02 * mse_ref


def test_k8v4_append_onto_prebuilt_cache():
    """7B-like cache: 32 layers x 8192 tokens x 8 heads prebuilt (K int8, V int4), then three single-token
    appends at t = 8192, 8193, 8194 of a 9216-token cache; earlier rows must not change."""
    w = I.K8V4
    n_outer, T, H, d, t_cap = w.n_outer, w.tokens, w.kv_heads, w.d, w.t_cap
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    sk, sv = K.alloc_side(n_outer, t_cap, H, d, 8, 16), K.alloc_side(n_outer, t_cap, H, d, 4, 16)
    sk.x, sv.x = xk, xv
    K.srft_kv_quantize(sk, sv, n_outer, T, H, d, 16, t_cap, 0, w.sign_seed)
    torch.cuda.synchronize()
    before_k = sk.codes[:, :, :T].clone()
    before_v = sv.scales[:, :, :T].clone()
    g = torch.Generator(device="cuda").manual_seed(44)
    new = []
    for step in range(3):
        nk = torch.randn((n_outer, 1, H, d), generator=g, device="cuda").half()
        nv = torch.randn((n_outer, 1, H, d), generator=g, device="cuda").half()
        ak, av = K.Side(sk.codes, sk.scales, 8, x=nk), K.Side(sv.codes, sv.scales, 4, x=nv)
        K.srft_kv_quantize(ak, av, n_outer, 1, H, d, 16, t_cap, T + step, w.sign_seed)
        new.append((nk, nv))
    torch.cuda.synchronize()
    assert torch.equal(before_k, sk.codes[:, :, :T]) and torch.equal(before_v, sv.scales[:, :, :T])
    for step, (nk, nv) in enumerate(new):
        for side, x, bits in ((sk, nk, 8), (sv, nv, 4)):
            enc = O.srft_kv_quantize(_np(x).astype(np.float64), None, bits, 16, w.sign_seed)
            assert_scales(_np(tm(side.scales)[:, T + step : T + step + 1]), enc["scales"])
            assert_codes(_np(tm(side.codes)[:, T + step : T + step + 1]), enc["r"], bits)
    # sampled prefix rows against the oracle
    rows = _sample_rows(n_outer * T * H, 1000, 45)
    for side, x, bits in ((sk, xk, 8), (sv, xv, 4)):
        xs = _np(x.reshape(-1, d)[rows]).astype(np.float64)
        enc = O.srft_kv_quantize(xs, None, bits, 16, w.sign_seed)
        o_idx, rem = rows // (T * H), rows % (T * H)
        crow = torch.as_tensor((o_idx * H + rem % H) * t_cap + rem // H, device="cuda")
        assert_codes(_np(side.codes.reshape(-1, d * bits // 8)[crow]), enc["r"], bits)
        assert_scales(_np(side.scales.reshape(-1, d // 16)[crow]), enc["scales"])


# ---------------------------------------------------------------------------
# the warp-per-vector quantize (d = 128 small calls, e.g. token appends)
# ---------------------------------------------------------------------------
WARP_CASES = [(bk, bv, g, lam) for bk, bv in ((4, 4), (8, 4), (4, 8), (8, 8)) for g in (16, 32) for lam in (False, True)]


@pytest.mark.parametrize("bk,bv,group,lam", WARP_CASES)
def test_warp_quantize_path(monkeypatch, bk, bv, group, lam):
    """One warp per vector (forced): 2 outer x 37 tokens x 3 heads written at t_offset 5 of t_cap 50, K and V of
    different widths in one launch, rows outside the window untouched."""
    monkeypatch.setenv("SRFTKV_QUANT_PATH", "warp")
    w = I.Workload("warp", n_outer=2, tokens=37, kv_heads=3, d=128, lam=lam, data_seed=bk * 10 + bv + group,
                   outlier_kind="scale", outlier_channels=4, outlier_factor=50.0)
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    lk, lv = I.lam_table(w, "k"), I.lam_table(w, "v")
    sk, sv = _quantize_gpu(xk, xv, lk, lv, bk, bv, group, 17, t_cap=50, t_offset=5)
    for side, x, lam_t, b in ((sk, xk, lk, bk), (sv, xv, lv, bv)):
        _check_side(side, x, lam_t, b, group, 17, t_offset=5)
        codes = _np(tm(side.codes))
        assert (codes[:, :5] == 0xAB).all() and (codes[:, 42:] == 0xAB).all(), "rows outside the window were written"


@pytest.mark.parametrize("transform,fmt", (("srht", "fp32"), ("srht", "e8m0"), ("srft", "fp16"), ("srft", "e8m0")))
@pytest.mark.parametrize("bits", (4, 8))
def test_warp_quantize_transforms_and_formats(monkeypatch, transform, fmt, bits):
    """The warp path with the Hadamard transform and the fp16 / e8m0 scale planes (stored scales bit-exact away
    from a rounding boundary of the format, codes against the stored scale)."""
    from tests.test_gpu_scale_formats import near_boundary, raw_np

    monkeypatch.setenv("SRFTKV_QUANT_PATH", "warp")
    n, T, H, g, seed = 2, 64, 4, 16, 23
    w = I.Workload("warpf", n_outer=n, tokens=T, kv_heads=H, d=128, lam=True, data_seed=bits + len(fmt),
                   outlier_kind="scale", outlier_channels=2, outlier_factor=30.0)
    x, lam = I.kv_side(w, "k"), I.lam_table(w, "k")
    s = K.alloc_side(n, T, H, 128, bits, g, transform=transform, scale_format=fmt)
    s.x, s.lam = x.cuda(), lam.cuda()
    K.srft_kv_quantize(s, None, n, T, H, 128, g, T, 0, seed)
    torch.cuda.synchronize()
    enc = O.srft_kv_quantize(_np(x).astype(np.float64), _np(lam)[:, None, :, :], bits, g, seed, transform=transform,
                             scale_format=fmt)
    raw = raw_np(s.scales, fmt) if fmt != "fp32" else _np(tm(s.scales))
    if fmt == "fp32":
        assert_scales(raw, enc["scales"])
        assert_codes(_np(tm(s.codes)), enc["r"], bits)
    else:
        want = np.asarray(enc["scales_raw"])
        diff = raw != want
        assert not (diff & ~near_boundary(enc["a_over_q"], fmt)).any()
        sc = np.repeat(O.decode_scales(raw, fmt), g, axis=-1)
        assert_codes(_np(tm(s.codes)), np.where(sc > 0, enc["z"] / np.where(sc > 0, sc, 1.0), 0.0), bits)


def test_warp_path_matches_tensor_core_path(monkeypatch):
    """The same 1000 vectors through the warp kernel and the tensor-core kernel: scales agree to 1e-5 and codes
    agree except at rounding ties (both are checked against the oracle elsewhere)."""
    n, T, H, g = 1, 250, 4, 16
    w = I.Workload("cmp", n_outer=n, tokens=T, kv_heads=H, d=128, data_seed=77)
    x = I.kv_side(w, "k")
    outs = {}
    for path in ("warp", "tc"):
        monkeypatch.setenv("SRFTKV_QUANT_PATH", path)
        s = K.alloc_side(n, T, H, 128, 4, g)
        s.x = x.cuda()
        K.srft_kv_quantize(s, None, n, T, H, 128, g, T, 0, 5)
        torch.cuda.synchronize()
        outs[path] = (_np(s.codes), _np(s.scales))
    assert np.allclose(outs["warp"][1], outs["tc"][1], rtol=1e-5, atol=0)
    qa, qb = O.unpack_codes(outs["warp"][0], 4), O.unpack_codes(outs["tc"][0], 4)
    assert (np.abs(qa - qb) <= 1).all() and (qa != qb).mean() < 1e-3
