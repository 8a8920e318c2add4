"""The device give-up paths of the attention kernel and of the register-path
quantize kernels, on the GPU, without a fault.

Every wait of the library's kernels on an asynchronous copy is bounded; a
warp of the attention split kernel that gives up sets bit 8 of the fault word,
waits (with the normal bound) for its own copies in flight, and contributes
an empty partial.  The test hook srftkv_set_attention_poll_limit_for_testing
shortens only the chunk wait, so that every warp gives up at its first chunk
while every copy it issued still lands: the call must finish, leave the fault
word set (and clear it when read), write the empty result (zeros), and leave
the context usable, so that the next call with the default limit is bitwise
the one before.  srftkv_set_codec_poll_limit_for_testing does the same for
the quantize kernels that stream x by asynchronous copies (the
one-thread-per-vector FFT kernel of d <= 128, the two-lane kernel of d = 192
and 256, and the MMA-issuing thread of the d = 128 tensor-core kernel, which
then issues no MMA while the epilogue warps' own waits run out): bit 0 of
the fault word, no code or scale stored, and the next call bitwise the call
before.
"""

import numpy as np
import pytest
import torch

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
    K.srftkv_set_attention_poll_limit_for_testing(-1)
    K.srftkv_set_codec_poll_limit_for_testing(-1)
    assert K.srftkv_device_fault() == 0


@pytest.mark.parametrize("d", (128, 80))
@pytest.mark.parametrize("static", (False, True))
def test_attention_gives_up_cleanly(d, static):
    import tests.test_gpu_attention as TA

    TA.K = K
    B, Hkv, rep, t_cap, seed = 2, 2, 4, 512, 9
    Hq = Hkv * rep
    sk, sv = TA.build_cache(B, Hkv, d, t_cap, 4, 4, 16, seed, data_seed=d)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hq, data_seed=d + 1), device="cuda")
    seq = torch.tensor([512, 300], dtype=torch.int32, device="cuda")
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, t_cap, 0), dtype=torch.uint8,
                     device="cuda")

    def call():
        out.fill_(float("nan"))
        if static:
            K.q4kv_decode_attention_static(q, out, sk, sv, B, Hq, Hkv, d, 16, t_cap, seq, 0.0, seed, 0)
        else:
            K.q4kv_decode_attention(q, out, sk, sv, B, Hq, Hkv, d, 16, t_cap, seq, 0.0, seed, 0, ws)
        torch.cuda.synchronize()
        return out.clone()

    assert K.srftkv_device_fault() == 0
    before = call()
    ref = TA.oracle_attention(q, sk, sv, 16, seed, seq)
    assert np.abs(before.cpu().numpy() - ref).max() <= ATTN_ATOL
    assert K.srftkv_device_fault() == 0
    try:
        K.srftkv_set_attention_poll_limit_for_testing(0)
        gave_up = call()
    finally:
        K.srftkv_set_attention_poll_limit_for_testing(-1)
    fault = K.srftkv_device_fault()
    assert fault & (1 << 8), f"fault word {fault:#x}: the attention bit is not set"
    assert fault & 0xFF == 0, "the codec's bit is set"
    assert K.srftkv_device_fault() == 0, "reading the fault word clears it"
    assert torch.equal(gave_up, torch.zeros_like(gave_up)), "a call whose warps all gave up writes zeros"
    after = call()
    assert K.srftkv_device_fault() == 0
    assert torch.equal(after, before), "the context is usable and the result unchanged after a give-up"


# (d, forced path): d = 128 forced onto the one-thread-per-vector FFT kernel (a call this small would
# otherwise take the one-warp-per-vector kernel, which has no asynchronous copies) and onto the tensor-core
# kernel; at d = 192 and 256 a call this small takes the two-lane register kernel by itself
@pytest.mark.parametrize("d,path", [(128, "fft"), (128, "tc"), (192, None), (256, None)])
def test_quantize_gives_up_cleanly(d, path, monkeypatch):
    if path is not None:
        monkeypatch.setenv("SRFTKV_QUANT_PATH", path)
    w = I.Workload("give_up", n_outer=2, tokens=300, kv_heads=2, d=d, data_seed=d)
    B, T, H, G, seed = w.n_outer, w.tokens, w.kv_heads, w.group, 5
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    sk, sv = K.alloc_side(B, T, H, d, 4, G), K.alloc_side(B, T, H, d, 4, G)
    sk.x, sv.x = xk, xv

    def call():
        for side in (sk, sv):
            side.codes.fill_(0xA5)
            side.scales.view(torch.uint8).fill_(0x5A)
        K.srft_kv_quantize(sk, sv, B, T, H, d, G, T, 0, seed)
        torch.cuda.synchronize()
        return [t.clone() for t in (sk.codes, sk.scales, sv.codes, sv.scales)]

    assert K.srftkv_device_fault() == 0
    before = call()
    assert K.srftkv_device_fault() == 0
    assert not torch.equal(before[0], torch.full_like(before[0], 0xA5)), "the reference call stored nothing"
    try:
        K.srftkv_set_codec_poll_limit_for_testing(0)
        gave_up = call()
    finally:
        K.srftkv_set_codec_poll_limit_for_testing(-1)
    fault = K.srftkv_device_fault()
    assert fault & 1, f"fault word {fault:#x}: the codec bit is not set"
    assert not fault & (1 << 8), "the attention bit is set"
    assert K.srftkv_device_fault() == 0, "reading the fault word clears it"
    for t in gave_up[0::2]:
        assert torch.equal(t, torch.full_like(t, 0xA5)), "a warp that gave up stored codes"
    for t in gave_up[1::2]:
        raw = t.view(torch.uint8)
        assert torch.equal(raw, torch.full_like(raw, 0x5A)), "a warp that gave up stored scales"
    after = call()
    assert K.srftkv_device_fault() == 0
    for a, b in zip(after, before):
        assert torch.equal(a, b), "the context is usable and the result unchanged after a give-up"
