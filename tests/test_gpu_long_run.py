"""GPU parity of decode attention over one long run of chunks per warp.

With n_splits = 1 the one CTA of a (sequence, kv head) streams the whole
context and each of its four warps a quarter of it (32768 tokens at
T = 131072).  That is where the code offset the V-side MMAs accumulate
((code + offset) * B, the offset removed with the column sums of B) would grow
largest before it cancels; the kernel folds it out every 64 chunks.  Checked
against the fp64 oracle on the same quantised cache ([GEM] Flash Attention
section: the online softmax over tiles equals softmax attention; [WQF]
Methodology 1: scores and outputs in the rotated domain), and against the
automatic split count, whose warps run about 50 chunks each: the split count
must not change the result beyond fp32 rounding.
"""

import math

import numpy as np
import pytest
import torch

from oracle import srft_oracle as O
from int8_kv_cache_srft_gb300 import inputs as I
from tests.parity import ATTN_ATOL

pytestmark = pytest.mark.gpu

K = None
SPLIT_ATOL = 2e-4  # one split against the automatic count (measured about 2e-5; the unfolded offset drifted by 1e-2)


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


@pytest.mark.parametrize("d", [128, 96])
def test_one_split_over_a_long_context(d):
    w = I.DECODE.resized(n_outer=1, kv_heads=2, q_heads=8, d=d)
    B, Hkv, T, Hq, G, seed = w.n_outer, w.kv_heads, w.tokens, w.q_heads, w.group, w.sign_seed
    rep = Hq // Hkv
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    sk, sv = K.alloc_side(B, T, Hkv, d, 4, G), K.alloc_side(B, T, Hkv, d, 4, G)
    sk.x, sv.x = xk, xv
    K.srft_kv_quantize(sk, sv, B, T, Hkv, d, G, T, 0, seed)
    q = I.query(w, device="cuda")
    outs = {}
    for ns in (1, 0):
        out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
        ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, T, ns), dtype=torch.uint8,
                         device="cuda")
        K.q4kv_decode_attention(q, out, sk, sv, B, Hq, Hkv, d, G, T, None, 0.0, seed, ns, ws)
        torch.cuda.synchronize()
        outs[ns] = _np(out).astype(np.float64)
    assert np.abs(outs[1] - outs[0]).max() <= SPLIT_ATOL
    qn = _np(q).astype(np.float64)
    for h in range(Hkv):
        kh = O.srft_kv_dequantize(_np(sk.codes[0, h]), _np(sk.scales[0, h]).astype(np.float64), None, 4, G, seed)
        vh = O.srft_kv_dequantize(_np(sv.codes[0, h]), _np(sv.scales[0, h]).astype(np.float64), None, 4, G, seed)
        for r in range(rep):
            hq = h * rep + r
            s = kh @ qn[0, hq] / math.sqrt(d)
            pw = np.exp(s - s.max())
            ref = (pw @ vh) / pw.sum()
            for ns in (1, 0):
                assert np.abs(outs[ns][0, hq] - ref).max() <= ATTN_ATOL, (ns, hq)
