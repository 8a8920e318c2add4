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


@pytest.mark.parametrize("rep", (5, 6, 8, 16))
@pytest.mark.parametrize("bk,bv", ((4, 4), (8, 4), (16, 16)))
@pytest.mark.parametrize("n_splits", (0, 3))
def test_attention_gqa_head_groups(rep, bk, bv, n_splits):
    """GQA ratios above four run as head groups of at most four query heads (5 -> 3 + 2, 6 -> 3 + 3, 8 -> 4 + 4,
    16 -> 4 x 4): every query head against the oracle, ragged sequence lengths."""
    B, Hkv, d, t_cap, seed = 2, 2, 128, 700, 12
    Hq = Hkv * rep
    sk, sv = build_cache(B, Hkv, d, t_cap, bk, bv, 16, seed, lam=(bk != 16), data_seed=rep * 7 + bk)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hq, data_seed=rep + 90), device="cuda")
    seq = torch.tensor([700, 333], dtype=torch.int32, device="cuda")
    out = run_attention(q, sk, sv, B, Hq, Hkv, d, 16, t_cap, seq, seed, n_splits=n_splits)
    ref = oracle_attention(q, sk, sv, 16, seed, seq)
    assert np.abs(out - ref).max() <= ATTN_ATOL


@pytest.mark.parametrize("d", (64, 80, 96, 192, 256))
def test_attention_gqa8_other_head_dims(d):
    B, Hkv, rep, t_cap, seed = 2, 1, 8, 320, 13
    Hq = Hkv * rep
    sk, sv = build_cache(B, Hkv, d, t_cap, 4, 4, 16, seed, data_seed=d + 3)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hq, data_seed=d + 4), device="cuda")
    seq = torch.tensor([320, 45], dtype=torch.int32, device="cuda")
    out = run_attention(q, sk, sv, B, Hq, Hkv, d, 16, t_cap, seq, seed)
    ref = oracle_attention(q, sk, sv, 16, seed, seq)
    assert np.abs(out - ref).max() <= ATTN_ATOL


def _quantize(x, bits, group, seed, lam=None, scale_format="fp32"):
    B, T, H, d = x.shape
    s = K.alloc_side(B, T, H, d, bits, group, scale_format=scale_format)
    s.x, s.lam = x, lam
    K.srft_kv_quantize(s, None, B, T, H, d, group, T, 0, seed)
    torch.cuda.synchronize()
    return s


@pytest.mark.parametrize("k", (10, 14, -20))
@pytest.mark.parametrize("bits_v,fmt", ((4, "fp32"), (8, "fp32"), (4, "e8m0")))
def test_value_scales_far_from_one(k, bits_v, fmt):
    """V scales far outside [2^-13, 2^7): a per-channel lambda_V = 2^k multiplies every rotated V coordinate
    (k = 10 gives |z_V| near 5000 and 4-bit scales near 700, past the 255 at which p * scale_V would overflow
    fp16; k = -20 gives scales near 1e-6).  The codes are those of lambda = 1 and the scales 2^k times larger
    (an exact power-of-two scaling), and attention divides by lambda_V, so the output must be that of the
    lambda = 1 cache, and within the tolerance of the oracle on the same cache."""
    B, Hkv, rep, d, T, seed = 2, 2, 4, 128, 600, 17
    Hq = Hkv * rep
    w = I.Workload("vrange", n_outer=B, tokens=T, kv_heads=Hkv, d=d, data_seed=41)
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    sk = _quantize(xk, 4, 16, seed)
    sv1 = _quantize(xv, bits_v, 16, seed, scale_format=fmt)
    lam = torch.full((1, Hkv, d), 2.0**k, dtype=torch.float32, device="cuda")
    svk = _quantize(xv, bits_v, 16, seed, lam=lam, scale_format=fmt)
    assert torch.equal(svk.codes, sv1.codes)
    if fmt == "fp32":
        assert torch.equal(svk.scales, sv1.scales * 2.0**k)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hq, data_seed=42), device="cuda")
    seq = torch.tensor([600, 211], dtype=torch.int32, device="cuda")
    o1 = run_attention(q, sk, sv1, B, Hq, Hkv, d, 16, T, seq, seed)
    ok = run_attention(q, sk, svk, B, Hq, Hkv, d, 16, T, seq, seed)
    assert np.isfinite(ok).all()
    assert np.abs(ok - o1).max() <= 1e-5 * max(1.0, float(np.abs(o1).max()))
    if fmt == "fp32":
        ref = oracle_attention(q, sk, svk, 16, seed, seq)
        assert np.abs(ok - ref).max() <= ATTN_ATOL


def test_value_magnitudes_scaled_by_1024():
    """V inputs times 2^10 (fp16 holds them exactly, |v| up to about 5000): codes unchanged, scales 2^10 times
    larger (near 700, past the old fp16 limit of 255), outputs 2^10 times the unscaled ones; against the oracle
    the 2e-3 rule is applied to the output divided by 2^10."""
    B, Hkv, rep, d, T, seed = 2, 2, 4, 128, 600, 18
    Hq = Hkv * rep
    w = I.Workload("vbig", n_outer=B, tokens=T, kv_heads=Hkv, d=d, data_seed=43)
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    sk = _quantize(xk, 4, 16, seed)
    sv1 = _quantize(xv, 4, 16, seed)
    svb = _quantize(xv * 1024.0, 4, 16, seed)
    assert torch.equal(svb.codes, sv1.codes) and torch.equal(svb.scales, sv1.scales * 1024.0)
    assert float(svb.scales.max()) > 255.0
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hq, data_seed=44), device="cuda")
    o1 = run_attention(q, sk, sv1, B, Hq, Hkv, d, 16, T, None, seed)
    ob = run_attention(q, sk, svb, B, Hq, Hkv, d, 16, T, None, seed)
    assert np.isfinite(ob).all()
    assert np.abs(ob / 1024.0 - o1).max() <= 1e-5 * max(1.0, float(np.abs(o1).max()))
    ref = oracle_attention(q, sk, svb, 16, seed, None)
    assert np.abs(ob - ref).max() / 1024.0 <= ATTN_ATOL


def test_value_scales_spanning_many_binades_across_chunks():
    """One cache whose V rows alternate, 64 tokens at a time, between magnitudes 2^13 and 2^-12 (fp16 inputs,
    a range of 2^25 in the scales): the V unit moves up and down between chunks.  Keys make the large rows'
    scores very low, so the small rows carry the output; checked against the oracle relative to the output's
    size."""
    B, Hkv, d, T, seed = 1, 1, 128, 512, 19
    w = I.Workload("vspan", n_outer=B, tokens=T, kv_heads=Hkv, d=d, data_seed=45)
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=1, data_seed=46), device="cuda")
    big = ((torch.arange(T, device="cuda") // 64) % 2 == 0)
    xv = torch.where(big[None, :, None, None], xv.float() * 2.0**13, xv.float() * 2.0**-12).half()
    qk = q.float()[:, None, :, :].expand(B, T, Hkv, d)
    xk = torch.where(big[None, :, None, None], -3.0 * qk, xk.float()).half()
    sk = _quantize(xk, 8, 16, seed)
    sv = _quantize(xv, 4, 16, seed)
    for n_splits in (1, 0):
        out = run_attention(q, sk, sv, B, 1, Hkv, d, 16, T, None, seed, n_splits=n_splits)
        ref = oracle_attention(q, sk, sv, 16, seed, None)
        assert np.isfinite(out).all()
        assert np.abs(out - ref).max() <= 1e-4 * float(np.abs(ref).max())


@pytest.mark.parametrize("bits", [4, 16])
def test_attention_captured_in_a_cuda_graph_matches_eager(bits):
    """The attention call (q preparation, split kernel and combine, the last two
    launched as programmatic dependents of the kernel before them) captured in a
    CUDA graph and replayed gives the eager call's output bit for bit, also
    after the query and the sequence lengths change in place between replays."""
    B, Hq, Hkv, d, T, G, seed = 3, 8, 2, 128, 2048, 16, 9
    sk, sv = build_cache(B, Hkv, d, T, bits, bits, G, seed)
    gen = torch.Generator(device="cuda").manual_seed(4)
    q = torch.randn((B, Hq, d), generator=gen, device="cuda").to(torch.float16)
    seq = torch.tensor([T, 1000, 17], dtype=torch.int32, device="cuda")
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, T, 0), dtype=torch.uint8, device="cuda")
    call = lambda: K.q4kv_decode_attention(q, out, sk, sv, B, Hq, Hkv, d, G, T, seq, 0.0, seed, 0, ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # the first call sets the kernels' attributes outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for step in range(3):
        if step:
            q.copy_(torch.randn((B, Hq, d), generator=gen, device="cuda").to(torch.float16))
            seq.copy_(torch.tensor([T - 7 * step, 1 + 300 * step, 2048 - 500 * step], dtype=torch.int32))
        call()
        torch.cuda.synchronize()
        eager = out.clone()
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager), step


@pytest.mark.parametrize("group,rep,n_splits", [(32, 3, 0), (64, 4, 3), (16, 3, 1)])
def test_d256_q_fragments_in_shared_memory(group, rep, n_splits):
    """d = 256 with 4-bit keys keeps q's K-side fragments in shared memory: the generic-group instance (groups
    32 and 64), a head group of three query heads (the fourth column padded) and single or few splits, with
    lambda on both sides, against the oracle on the same quantised cache."""
    B, Hkv, d, t_cap, seed = 2, 2, 256, 520, 13
    Hq = Hkv * rep
    sk, sv = build_cache(B, Hkv, d, t_cap, 4, 4, group, seed, lam=True, data_seed=group + rep)
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hq, data_seed=group * rep),
                device="cuda")
    seq = torch.tensor([520, 77], dtype=torch.int32, device="cuda")
    out = run_attention(q, sk, sv, B, Hq, Hkv, d, group, t_cap, seq, seed, n_splits=n_splits)
    ref = oracle_attention(q, sk, sv, group, seed, seq)
    assert np.abs(out - ref).max() <= ATTN_ATOL
