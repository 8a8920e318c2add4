"""q4kv_decode_attention_static: decode attention for callers that cannot
allocate device memory (a runtime whose memory is all in its own pool, a
plugin without access to its host's allocator, code that cannot take
cudaMalloc's implicit synchronisation).  It uses the library's fixed-size
device array as scratch instead of a caller workspace.

Checked through the C ABI against q4kv_decode_attention with a caller
workspace, on two calls in a row (the array keeps the previous call's
contents).  Both run the same kernels with the same split count, so the
outputs must be identical bit for bit; a partial result read from stale or
misplaced scratch could hide inside a tolerance.  Also checked: the automatic
split count is lowered until the workspace fits the array, and sizes beyond
the array are rejected.  This file is
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
        assert bool(torch.isfinite(got).all())
        assert torch.equal(got, ref), f"call {call}: static scratch and caller workspace outputs differ"
        outs.append(got.cpu().numpy())
    assert np.abs(outs[0] - outs[1]).max() > 0  # the second call really recomputed
    assert K.srftkv_device_fault() == 0


def test_static_scratch_lowers_the_automatic_split_count_to_fit(K):
    """B=64, Hq=32, Hkv=8, d=256, t_cap=2048: the automatic split count on a 152-SM GB300 (8) needs about
    19 MB of workspace, more than the array; the static entry lowers it to the largest count that fits and gives
    exactly the workspace entry's output at that count."""
    B, Hkv, rep, d, T, seed = 64, 8, 4, 256, 2048, 9
    Hq = Hkv * rep
    cap = K.STATIC_SCRATCH_BYTES
    auto = K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, T, 0)
    fit = max(n for n in range(1, 65) if K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, T, n) <= cap)
    sk, sv = _cache(K, B, Hkv, d, T, seed, 73)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hq, data_seed=73), device="cuda")
    seq = I.seq_lens(B, T, 73, device="cuda")
    ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, T, fit), dtype=torch.uint8, device="cuda")
    ref = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    got = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
    K.q4kv_decode_attention(q, ref, sk, sv, B, Hq, Hkv, d, 16, T, seq, 0.0, seed, fit, ws)
    K.q4kv_decode_attention_static(q, got, sk, sv, B, Hq, Hkv, d, 16, T, seq, 0.0, seed, 0)
    torch.cuda.synchronize()
    if auto > cap:  # the case this test is about (152 SMs); on a smaller GPU the automatic count may fit already
        assert torch.equal(got, ref)
    else:
        assert float((got - ref).abs().max()) <= ATTN_ATOL
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
