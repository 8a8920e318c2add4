"""q4kv_decode_attention_static: decode attention for callers that cannot
allocate device memory (a runtime whose memory is all in its own pool, a
plugin without access to its host's allocator, code that cannot take
cudaMalloc's implicit synchronisation).  It uses the library's fixed-size
device array as scratch instead of a caller workspace.

Checked through the C ABI against q4kv_decode_attention with a caller
workspace, on two calls in a row (the array keeps the previous call's
contents), plus the rejection of sizes beyond the array.  This file is
collected last on purpose and is self-contained, so it passes both alone and
after the other GPU tests.
"""

import numpy as np
import pytest
import torch

from int8_kv_cache_srft_gb300 import inputs as I
from tests.parity import ATTN_ATOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import int8_kv_cache_srft_gb300 as mod

    mod.library()
    return mod


def _cache(K, B, Hkv, d, T, seed, data_seed):
    w = I.Workload("noalloc", n_outer=B, tokens=T, kv_heads=Hkv, d=d, data_seed=data_seed)
    sk, sv = K.alloc_side(B, T, Hkv, d, 4, 16), K.alloc_side(B, T, Hkv, d, 4, 16)
    sk.x, sv.x = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    K.srft_kv_quantize(sk, sv, B, T, Hkv, d, 16, T, 0, seed)
    return sk, sv


def test_static_scratch_matches_workspace_entry_point_twice(K):
    B, Hkv, rep, d, T, seed = 4, 8, 4, 128, 4096, 5
    Hq = Hkv * rep
    seq = torch.tensor([4096, 1000, 1, 2500], dtype=torch.int32, device="cuda")
    outs = []
    for call, data_seed in enumerate((71, 72)):  # two calls in a row on different data
        sk, sv = _cache(K, B, Hkv, d, T, seed, data_seed)
        q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hq, data_seed=data_seed),
                    device="cuda")
        ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, T, 0), dtype=torch.uint8, device="cuda")
        ref = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
        got = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
        K.q4kv_decode_attention(q, ref, sk, sv, B, Hq, Hkv, d, 16, T, seq, 0.0, seed, 0, ws)
        K.q4kv_decode_attention_static(q, got, sk, sv, B, Hq, Hkv, d, 16, T, seq, 0.0, seed, 0)
        torch.cuda.synchronize()
        r, g = ref.cpu().numpy(), got.cpu().numpy()
        assert np.isfinite(g).all()
        assert np.abs(g - r).max() <= ATTN_ATOL
        outs.append(g)
    assert np.abs(outs[0] - outs[1]).max() > 0  # the second call really recomputed
    assert K.srftkv_device_fault() == 0


def test_static_scratch_rejects_sizes_beyond_the_array(K):
    B, Hkv, rep, d, T = 16, 8, 4, 128, 1 << 20
    Hq = Hkv * rep
    n_splits = 4096
    assert K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, T, n_splits) > K.STATIC_SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    side = K.Side(dummy, torch.empty(4, dtype=torch.float32, device="cuda"), 4)
    q = torch.empty((B, Hq, d), dtype=torch.float16, device="cuda")
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    with pytest.raises(K.SrftKvError) as e:
        K.q4kv_decode_attention_static(q, out, side, side, B, Hq, Hkv, d, 16, T, None, 0.0, 1, n_splits)
    assert e.value.code == K.SRFTKV_ERR_INVALID
    assert "static array" in str(e.value)
