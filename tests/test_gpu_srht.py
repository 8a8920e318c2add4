"""GPU parity of the Hadamard variant (SRHT = d^-1/2 H diag(s) x, Sylvester
natural order) against the fp64 oracle: the bare transform, the codec on
both kernel paths (the register transform for every d, the tensor-core
contraction for d = 128), a call whose K and V sides use different
transforms, and decode attention over SRHT-rotated caches."""

import numpy as np
import pytest
import torch

from oracle import srft_oracle as O
from int8_kv_cache_srft_gb300 import inputs as I
from tests.parity import ATTN_ATOL, assert_codes, assert_dequant_within_step, assert_reconstruction_bound, assert_scales

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
    return t.permute(0, 2, 1, 3)


@pytest.mark.parametrize("d", (16, 32, 64, 128, 256))
@pytest.mark.parametrize("inverse", (False, True))
def test_srht_transform_matches_oracle(d, inverse):
    g = torch.Generator().manual_seed(50 + d)
    n = 777
    x = (torch.randn((n, d), generator=g) * 3).to(torch.float16)
    y = torch.empty((n, d), dtype=torch.float32, device="cuda")
    K.srht_transform(x.cuda(), y, n, d, 5, inverse)
    torch.cuda.synchronize()
    xd = _np(x).astype(np.float64)
    ref = O.srht_inverse(xd, 5) if inverse else O.srht_forward(xd, 5)
    err = np.abs(_np(y) - ref).max(axis=-1)
    assert np.all(err <= 2e-6 * np.linalg.norm(xd, axis=-1) + 1e-7)


def _encode(w, tr_k, tr_v, bits_k, bits_v, group, seed, t_cap, t_offset):
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    lk, lv = I.lam_table(w, "k"), I.lam_table(w, "v")
    n, T, H, d = xk.shape
    sides = []
    for x, lam, bits, tr in ((xk, lk, bits_k, tr_k), (xv, lv, bits_v, tr_v)):
        s = K.alloc_side(n, t_cap, H, d, bits, group, transform=tr)
        s.codes.fill_(0xAB)
        s.scales.fill_(-1.0)
        s.x = x.cuda()
        s.lam = None if lam is None else lam.cuda()
        sides.append(s)
    K.srft_kv_quantize(sides[0], sides[1], n, T, H, d, group, t_cap, t_offset, seed)
    torch.cuda.synchronize()
    return sides, (xk, xv), (lk, lv)


def _check(side, x, lam, bits, group, seed, tr, t_offset):
    n, T, H, d = x.shape
    lam_b = None if lam is None else _np(lam)[:, None, :, :]
    enc = O.srft_kv_quantize(_np(x).astype(np.float64), lam_b, bits, group, seed, transform=tr)
    assert_scales(_np(tm(side.scales))[:, t_offset:t_offset + T], enc["scales"])
    assert_codes(_np(tm(side.codes))[:, t_offset:t_offset + T], enc["r"], bits)
    out = torch.empty_like(side.x)
    K.srft_kv_dequantize(K.Side(side.codes, side.scales, bits, x=out, lam=side.lam, transform=tr), None, n, T, H, d,
                         group, side.codes.shape[2], t_offset, seed)
    torch.cuda.synchronize()
    lam_full = None if lam_b is None else np.broadcast_to(lam_b, x.shape)
    ref_hat = O.srft_kv_dequantize(enc["codes"], enc["scales"], lam_b, bits, group, seed, transform=tr)
    assert_dequant_within_step(_np(out), ref_hat, enc["scales"], lam_full, group)
    assert_reconstruction_bound(_np(out), _np(x), enc["scales"], lam_full, group)


@pytest.mark.parametrize("d,bits,path", [(d, b, p) for d in (16, 32, 64, 128, 256) for b in (4, 8) for p in ("fft", "tc")
                                          if p == "fft" or d == 128])  # the tensor-core path is d = 128
def test_srht_codec(monkeypatch, d, bits, path):
    monkeypatch.setenv("SRFTKV_QUANT_PATH", path)
    w = I.Workload("srht", n_outer=2, tokens=261, kv_heads=3, d=d, lam=(bits == 4), data_seed=7 * d + bits,
                   outlier_kind="scale", outlier_channels=2, outlier_factor=30.0)
    (sk, sv), (xk, xv), (lk, lv) = _encode(w, "srht", "srht", bits, 12 - bits, 16, 17, t_cap=270, t_offset=4)
    _check(sk, xk, lk, bits, 16, 17, "srht", 4)
    _check(sv, xv, lv, 12 - bits, 16, 17, "srht", 4)


@pytest.mark.parametrize("d", (64, 128))
def test_mixed_transforms_in_one_call(d):
    """K rotated by the SRFT, V by the SRHT, in one quantize call (the host splits it for the tensor-core path)."""
    w = I.Workload("mixed", n_outer=2, tokens=300, kv_heads=2, d=d, data_seed=d)
    (sk, sv), (xk, xv), _ = _encode(w, "srft", "srht", 4, 4, 16, 23, t_cap=300, t_offset=0)
    _check(sk, xk, None, 4, 16, 23, "srft", 0)
    _check(sv, xv, None, 4, 16, 23, "srht", 0)


def _oracle_side(s, group):
    return {"bits": s.bits, "codes": _np(tm(s.codes)), "scales": _np(tm(s.scales)).astype(np.float64),
            "lam": None if s.lam is None else _np(s.lam).astype(np.float64), "group": group, "transform": s.transform}


@pytest.mark.parametrize("tr_k,tr_v", (("srht", "srht"), ("srht", "srft"), ("srft", "srht")))
@pytest.mark.parametrize("d", (64, 128, 256))
def test_srht_attention(tr_k, tr_v, d):
    B, Hkv, rep, t_cap, seed = 2, 2, 4, 400, 29
    w = I.Workload("attn", n_outer=B, tokens=t_cap, kv_heads=Hkv, d=d, lam=True, data_seed=d + 3,
                   outlier_kind="scale", outlier_channels=2, outlier_factor=8.0)
    (sk, sv), _, _ = _encode(w, tr_k, tr_v, 4, 4, 16, seed, t_cap=t_cap, t_offset=0)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hkv * rep, data_seed=d), device="cuda")
    seq = torch.tensor([400, 151], dtype=torch.int32, device="cuda")
    out = torch.empty((B, Hkv * rep, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hkv * rep, Hkv, d, t_cap, 0), dtype=torch.uint8,
                     device="cuda")
    K.q4kv_decode_attention(q, out, sk, sv, B, Hkv * rep, Hkv, d, 16, t_cap, seq, 0.0, seed, 0, ws)
    torch.cuda.synchronize()
    ref = O.packed_decode_attention(_np(q).astype(np.float64), _oracle_side(sk, 16), _oracle_side(sv, 16), seed,
                                    _np(seq))
    assert np.abs(_np(out) - ref).max() <= ATTN_ATOL
