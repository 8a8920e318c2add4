"""GPU parity at the full size of the packed-cache decode workload, in the
launch configuration the benchmark times.

B=16 sequences, Hq=32, Hkv=8, d=128, T=131072 tokens, int4/int4, group 16,
fp32 scales, planes of t_cap = T + 64 rows (room for the benchmark's one-token
append): the whole cache (2 x 16.8 M head vectors, 4 GiB of fp16 per side, so
the last rows of sequence 15 sit just below byte offset 2^32) is quantised in
one launch, dequantised in one launch and attended in one launch with the
automatic split count.

Checked:
  * every row, on the GPU, by properties that hold at any size: rows
    [0, T) of every plane written and rows [T, t_cap) untouched; in every
    group the largest |code| is Q = 7 (the absmax element maps to +-Q, [WQF]
    Methodology 2, step 4); every dequantised vector within the orthogonality
    bound ||x_hat - x||_2 <= ||scale / 2||_2 of its input;
  * sampled rows against the fp64 oracle (codes, scales, dequantised vectors),
    including the last 128-row tile of sequence 15, kv head 7;
  * attention outputs of sampled (sequence, kv head) pairs against the oracle
    on the same quantised cache, and the same kernel on the raw fp16 cache.
"""

import math

import numpy as np
import pytest
import torch

from oracle import srft_oracle as O
from int8_kv_cache_srft_gb300 import inputs as I
from tests.parity import ATTN_ATOL, assert_codes, assert_dequant_within_step, assert_scales

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


def _max_abs_code_per_group(codes: torch.Tensor, group: int) -> torch.Tensor:
    """Largest |q| per group of int4 code rows [..., d/2] (two's-complement nibbles, even coordinate low)."""
    lo = (codes & 0xF).to(torch.int16)
    hi = (codes >> 4).to(torch.int16)
    lo = torch.where(lo > 7, lo - 16, lo).abs()
    hi = torch.where(hi > 7, hi - 16, hi).abs()
    m = torch.maximum(lo, hi)  # per byte: coordinates 2j, 2j+1
    return m.reshape(*m.shape[:-1], -1, group // 2).amax(dim=-1)


def test_decode_workload_bench_launches_full_size():
    w = I.DECODE
    B, Hkv, d, T, Hq, G, seed = w.n_outer, w.kv_heads, w.d, w.tokens, w.q_heads, w.group, w.sign_seed
    rep = Hq // Hkv
    t_cap = T + 64
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    sk, sv = K.alloc_side(B, t_cap, Hkv, d, 4, G), K.alloc_side(B, t_cap, Hkv, d, 4, G)
    for s in (sk, sv):
        s.codes.fill_(0xAB)
        s.scales.fill_(-1.0)
    sk.x, sv.x = xk, xv
    K.srft_kv_quantize(sk, sv, B, T, Hkv, d, G, t_cap, 0, seed)
    ok_, ov_ = torch.empty_like(xk), torch.empty_like(xv)
    K.srft_kv_dequantize(K.Side(sk.codes, sk.scales, 4, x=ok_), K.Side(sv.codes, sv.scales, 4, x=ov_), B, T, Hkv, d,
                         G, t_cap, 0, seed)
    torch.cuda.synchronize()

    # ---- every row: properties that hold at any size (one sequence at a time) ----
    for side, x, xhat in ((sk, xk, ok_), (sv, xv, ov_)):
        assert bool((side.codes[:, :, T:] == 0xAB).all()), "rows past the written window were touched"
        assert bool((side.scales[:, :, T:] == -1.0).all()), "scale rows past the written window were touched"
        for b in range(B):
            sc = side.scales[b, :, :T]                      # [H][T][d/G]
            assert bool((sc > 0).all()), f"sequence {b}: unwritten or zero scale rows"
            assert bool((_max_abs_code_per_group(side.codes[b, :, :T], G) == 7).all()), \
                f"sequence {b}: a group whose largest |code| is not Q"
            err = (xhat[b].float() - x[b].float()).norm(dim=-1)          # [T][H]
            half_step = (sc.permute(1, 0, 2).double() / 2).repeat_interleave(G, dim=-1).norm(dim=-1)
            bound = half_step + xhat[b].float().norm(dim=-1).double() * 2.0**-11 + 1e-6
            assert bool((err.double() <= bound).all()), \
                f"sequence {b}: a vector outside the reconstruction bound (worst {float((err - bound).max()):.3g})"

    # ---- sampled rows against the oracle ----
    gen = np.random.default_rng(55)
    n_rand = 3000
    bs = gen.integers(0, B, n_rand)
    ts = gen.integers(0, T, n_rand)
    hs = gen.integers(0, Hkv, n_rand)
    tail = np.arange(T - 128, T)  # the last 128-row tile of (b = 15, kv head 7): fp16 offsets just below 2^32
    bs = np.concatenate([bs, np.full(tail.size, B - 1), [0, 0, B - 1]])
    ts = np.concatenate([ts, tail, [0, T - 1, 0]])
    hs = np.concatenate([hs, np.full(tail.size, Hkv - 1), [0, Hkv - 1, 0]])
    assert ((bs == B - 1) & (hs == Hkv - 1) & (ts == T - 1)).any()
    bi, ti, hi = (torch.from_numpy(a).cuda() for a in (bs, ts, hs))
    for side, x, xhat in ((sk, xk, ok_), (sv, xv, ov_)):
        xs = _np(x[bi, ti, hi]).astype(np.float64)[:, None, :]          # [n][1][d]
        enc = O.srft_kv_quantize(xs, None, 4, G, seed)
        codes = _np(side.codes[bi, hi, ti])[:, None, :]
        scales = _np(side.scales[bi, hi, ti])[:, None, :]
        assert_scales(scales, enc["scales"])
        assert_codes(codes, enc["r"], 4)
        got = _np(xhat[bi, ti, hi]).astype(np.float64)[:, None, :]
        # within one quantisation step of the oracle's decode of its own codes
        ref_hat = O.srft_kv_dequantize(enc["codes"], enc["scales"], None, 4, G, seed)
        assert_dequant_within_step(got, ref_hat, enc["scales"], None, G)
        # tight: against the oracle's decode of the GPU's codes
        mine = O.srft_kv_dequantize(codes, scales.astype(np.float64), None, 4, G, seed)
        assert np.abs(got - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5
    del ok_, ov_

    # ---- attention on the same cache: sampled (sequence, kv head) pairs ----
    q = I.query(w, device="cuda")
    seq = torch.full((B,), T, dtype=torch.int32, device="cuda")
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, t_cap, 0), dtype=torch.uint8,
                     device="cuda")
    K.q4kv_decode_attention(q, out, sk, sv, B, Hq, Hkv, d, G, t_cap, seq, 0.0, seed, 0, ws)
    rk, rv = xk.permute(0, 2, 1, 3).contiguous(), xv.permute(0, 2, 1, 3).contiguous()
    out16 = torch.empty_like(out)
    ws16 = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, T, 0), dtype=torch.uint8,
                       device="cuda")
    K.q4kv_decode_attention(q, out16, K.Side(rk, None, 16), K.Side(rv, None, 16), B, Hq, Hkv, d, G, T, None, 0.0,
                            seed, 0, ws16)
    torch.cuda.synchronize()
    del rk, rv
    out, out16 = _np(out), _np(out16)
    qn = _np(q).astype(np.float64)
    for b, h in ((0, 0), (B - 1, Hkv - 1), (7, 3)):
        kh = O.srft_kv_dequantize(_np(sk.codes[b, h, :T]), _np(sk.scales[b, h, :T]).astype(np.float64), None, 4, G,
                                  seed)
        vh = O.srft_kv_dequantize(_np(sv.codes[b, h, :T]), _np(sv.scales[b, h, :T]).astype(np.float64), None, 4, G,
                                  seed)
        k16, v16 = _np(xk[b, :, h]).astype(np.float64), _np(xv[b, :, h]).astype(np.float64)
        for r in range(rep):
            hq = h * rep + r
            for kk, vv, o in ((kh, vh, out), (k16, v16, out16)):
                s = kk @ qn[b, hq] / math.sqrt(d)
                pw = np.exp(s - s.max())
                ref = (pw @ vv) / pw.sum()
                assert np.abs(o[b, hq] - ref).max() <= ATTN_ATOL
