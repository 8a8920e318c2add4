"""GPU parity of packed-cache decode attention against the fp64 oracle.

The cache is quantised by the library's own quantize kernel; the oracle then
dequantises exactly those codes and scales and runs plain softmax attention,
so the comparison isolates the attention kernel (tolerance: 2e-3 max-abs).
"""

import numpy as np
import pytest
import torch

from oracle import srft_oracle as O
from int8_kv_cache_srft_gb300 import inputs as I
from tests.parity import ATTN_ATOL

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


def build_cache(B, Hkv, d, t_cap, bits_k, bits_v, group, seed, lam=False, data_seed=0, scale_outliers=True):
    """K/V sides quantised on the GPU (or raw fp16 for bits 16), plus the fp16 inputs."""
    w = I.Workload("attn", n_outer=B, tokens=t_cap, kv_heads=Hkv, d=d, lam=lam, data_seed=data_seed,
                   outlier_kind="scale" if scale_outliers else "none", outlier_channels=2, outlier_factor=8.0)
    sides = []
    for name, bits in (("k", bits_k), ("v", bits_v)):
        x = I.kv_side(w, name, device="cuda")
        lt = I.lam_table(w, name, device="cuda")
        if bits == 16:
            s = K.Side(x.permute(0, 2, 1, 3).contiguous(), None, 16)  # head-major raw cache
        else:
            s = K.alloc_side(B, t_cap, Hkv, d, bits, group)
            s.x, s.lam = x, lt
            K.srft_kv_quantize(s, None, B, t_cap, Hkv, d, group, t_cap, 0, seed)
        sides.append(s)
    torch.cuda.synchronize()
    return sides


def run_attention(q, sk, sv, B, Hq, Hkv, d, group, t_cap, seq_lens, seed, n_splits=0, sm_scale=0.0):
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, t_cap, n_splits), dtype=torch.uint8,
                     device="cuda")
    K.q4kv_decode_attention(q, out, sk, sv, B, Hq, Hkv, d, group, t_cap, seq_lens, sm_scale, seed, n_splits, ws)
    torch.cuda.synchronize()
    return _np(out)


def oracle_side(s, group, rows=None):
    """The oracle's token-major view [B][T][H][...] of a head-major side."""
    if s.bits == 16:
        v = _np(s.codes).transpose(0, 2, 1, 3)
        return {"bits": 16, "values": v if rows is None else v[rows]}
    codes, scales = _np(s.codes).transpose(0, 2, 1, 3), _np(s.scales).transpose(0, 2, 1, 3).astype(np.float64)
    lam = None if s.lam is None else _np(s.lam).astype(np.float64)
    if rows is not None:
        codes, scales = codes[rows], scales[rows]
        lam = None if lam is None else lam[rows]
    return {"bits": s.bits, "codes": codes, "scales": scales, "lam": lam, "group": group}


def oracle_attention(q, sk, sv, group, seed, seq_lens, sm_scale=None):
    ql = _np(q).astype(np.float64)
    L = None if seq_lens is None else _np(seq_lens)
    return O.packed_decode_attention(ql, oracle_side(sk, group), oracle_side(sv, group), seed, L, sm_scale)


CASES = []
for d in (64, 128, 256):
    for bk, bv in ((4, 4), (8, 4), (4, 8), (8, 8), (16, 16)):
        CASES.append((d, bk, bv))


@pytest.mark.parametrize("d,bk,bv", CASES)
def test_attention_matches_oracle_small(d, bk, bv):
    B, Hkv, rep, t_cap = 2, 2, 4, 300
    Hq = Hkv * rep
    seed = 21
    sk, sv = build_cache(B, Hkv, d, t_cap, bk, bv, 16, seed, lam=(bk != 16), data_seed=d + bk * 10 + bv)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hq, data_seed=d), device="cuda")
    seq = torch.tensor([300, 137], dtype=torch.int32, device="cuda")
    out = run_attention(q, sk, sv, B, Hq, Hkv, d, 16, t_cap, seq, seed)
    ref = oracle_attention(q, sk, sv, 16, seed, seq)
    err = np.abs(out - ref).max()
    assert err <= ATTN_ATOL, f"max-abs error {err:.3g}"


@pytest.mark.parametrize("rep", (1, 2, 3, 4))
@pytest.mark.parametrize("n_splits", (0, 1, 5))
def test_attention_gqa_and_splits(rep, n_splits):
    B, Hkv, d, t_cap, seed = 3, 2, 128, 1000, 8
    Hq = Hkv * rep
    sk, sv = build_cache(B, Hkv, d, t_cap, 4, 4, 16, seed, data_seed=rep)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hq, data_seed=rep + 50), device="cuda")
    seq = torch.tensor([1000, 1, 517], dtype=torch.int32, device="cuda")
    out = run_attention(q, sk, sv, B, Hq, Hkv, d, 16, t_cap, seq, seed, n_splits=n_splits, sm_scale=0.11)
    ref = oracle_attention(q, sk, sv, 16, seed, seq, sm_scale=0.11)
    assert np.abs(out - ref).max() <= ATTN_ATOL


def test_group32_and_full_length_default():
    B, Hkv, rep, d, t_cap, seed = 2, 1, 4, 128, 640, 4
    sk, sv = build_cache(B, Hkv, d, t_cap, 8, 4, 32, seed, lam=True)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=rep, data_seed=3), device="cuda")
    out = run_attention(q, sk, sv, B, rep, Hkv, d, 32, t_cap, None, seed)
    ref = oracle_attention(q, sk, sv, 32, seed, None)
    assert np.abs(out - ref).max() <= ATTN_ATOL


def test_zero_length_rows_and_split_invariance():
    B, Hkv, rep, d, t_cap, seed = 3, 2, 4, 128, 2048, 6
    sk, sv = build_cache(B, Hkv, d, t_cap, 4, 4, 16, seed)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hkv * rep, data_seed=9), device="cuda")
    seq = torch.tensor([0, 2048, 33], dtype=torch.int32, device="cuda")
    o1 = run_attention(q, sk, sv, B, Hkv * rep, Hkv, d, 16, t_cap, seq, seed, n_splits=1)
    oa = run_attention(q, sk, sv, B, Hkv * rep, Hkv, d, 16, t_cap, seq, seed, n_splits=0)
    o7 = run_attention(q, sk, sv, B, Hkv * rep, Hkv, d, 16, t_cap, seq, seed, n_splits=7)
    assert not o1[0].any() and not oa[0].any() and not o7[0].any()
    assert np.abs(o1 - oa).max() <= 1e-4 and np.abs(o1 - o7).max() <= 1e-4
    ref = oracle_attention(q, sk, sv, 16, seed, seq)
    assert np.abs(oa - ref).max() <= ATTN_ATOL


def test_raw_fp16_cache_ignores_garbage_past_sequence_end():
    B, Hkv, rep, d, t_cap, seed = 2, 2, 4, 128, 100, 1
    sk, sv = build_cache(B, Hkv, d, t_cap, 16, 16, 16, seed)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hkv * rep, data_seed=2), device="cuda")
    seq = torch.tensor([37, 100], dtype=torch.int32, device="cuda")
    ref = oracle_attention(q, sk, sv, 16, seed, seq)
    sk.codes[0, :, 37:] = float("nan")
    sv.codes[0, :, 37:] = float("inf")
    out = run_attention(q, sk, sv, B, Hkv * rep, Hkv, d, 16, t_cap, seq, seed)
    assert np.isfinite(out).all() and np.abs(out - ref).max() <= ATTN_ATOL
