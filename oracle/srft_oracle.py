"""fp64 CPU oracle for the SRFT KV-cache codec and packed-cache decode attention.

TEST INFRASTRUCTURE ONLY.  This module is the slow, obviously-correct
definition that the CUDA library is checked against.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the library itself never calls into it and has no CPU fallback.
It shares no code with the CUDA path: the only thing both sides consume is
the seeded synthetic input produced by ``int8_kv_cache_srft_gb300.inputs``.

Sources (page title, then section):

* [WQF] "When Quantization Is Free: An int4 KV Cache That Outruns fp16 on
  Apple Silicon" (summary page of arXiv 2605.05699), Methodology section 1
  (the SRFT definition SRFT(x) = pack(F . diag(s) . x), F the unitary DFT,
  s a fixed random sign vector), section 2 (the fused kernel's steps: sign
  multiply, radix-2 Stockham FFT of length d/2, Hermitian packing into a
  real representation, per-channel lambda rescale, per-group absmax, rounding
  to signed int4/int8, nibble packing) and section 3 (per-channel scaling
  combined with per-group scaling, groups of 16).
* [GEM] "Gemini on-device quantization, KV cache, Apple Silicon" (hotdry
  blog), section "INT8/INT4 quantization strategy" (the KV-memory formula
  2 x layers x kv_heads x head_dim x seq_len x dtype_bytes) and section
  "Flash Attention and Metal kernel fusion" (tiled attention with an online
  softmax; the softmax it computes is the plain one implemented here).
* [KVS] "Efficient LLM inference on Apple Silicon: KVSplit key techniques",
  sections "Key findings" (8-bit keys with 4-bit values, K8V4) and
  "Memory optimisation calculation" (the K8V4 byte formula).

Readings where the pages are silent (each is listed again in the design
notes; the CUDA path implements the same readings independently):

1. Sign vector: s_i = -1 when bit 63 of the splitmix64 output number i
   (counting from 0) of a generator seeded with ``sign_seed`` is set, else +1.
   splitmix64 is the published generator of Steele, Lea and Flood (OOPSLA
   2014), in the form popularised by Vigna.  One s per (seed, d), shared by K,
   V, q and every layer, head and token.
2. DFT sign: the forward transform uses exp(-2 pi i n k / d), scaled by
   d^(-1/2) (unitary).
3. Hermitian packing of the d/2+1 independent bins y_0..y_{d/2} of a real
   length-d input: p_0 = y_0, p_1 = y_{d/2} (both real),
   p_{2k} = sqrt(2) Re y_k, p_{2k+1} = sqrt(2) Im y_k for k = 1..d/2-1.
   With this scaling x -> p is an orthogonal real d x d map.
4. lambda multiplies the packed coordinate: z_i = lambda_i p_i.
5. Symmetric quantisation: Q = 2^(bits-1) - 1, scale_j = max_{i in G_j}
   |z_i| / Q, q_i = clamp(rint(z_i / scale_j), -Q, Q) with round-half-even;
   an all-zero group gets scale 0 and codes 0.  The codes -8 / -128 are
   never produced.
6. Nibble order: the even coordinate goes in the low nibble, two's
   complement.  int8 codes are stored as two's-complement bytes.
7. Attention softmax scale defaults to 1/sqrt(d); a query whose sequence
   length is 0 gets an all-zero output.
8. The Hadamard variant ([WQF] Methodology 1 names SRHT as the common
   alternative and Key results, quality, finds it indistinguishable from
   SRFT; the pages do not write it out): SRHT(x) = d^(-1/2) H diag(s) x with
   H the Sylvester Hadamard matrix in natural order, H_ij = (-1)^popcount(i & j),
   the same sign vector s as the SRFT, no subsampling and no packing (the
   output is already real).  Everything downstream (lambda, groups,
   rounding, packing, attention) is unchanged.
9. Lighter scale planes ([WQF] Key results, memory efficiency: 3.0-3.56x
   persistent compression, which fp32 scales cannot give).  The stored scale
   is what the codes are rounded against:
   - fp16: scale_j = A_j / Q rounded to the nearest fp16 (ties to even),
     saturating at 65504; q_i = clamp(rint(z_i / scale_j), -Q, Q).
   - e8m0 (one byte): scale_j = 2^e with e = ceil(log2(A_j / Q)) (the
     smallest power of two not below A_j / Q, so no code is clamped),
     e clamped to [-126, 127], stored as the byte e + 127.
   A zero group stores scale 0 (byte 0 for e8m0) and codes 0 in both.
   With int4 codes and groups of 16 this is 80 (fp16) and 72 (e8m0) bytes
   per d = 128 vector against 256 in fp16: 3.2x and 3.56x.
10. Head dimensions that are not powers of two ([WQF] Methodology 1: the
   SRFT's reason for being over the SRHT): the definitions above hold for
   any even d (the DFT has no power-of-two requirement; Hermitian packing
   needs d even).  The Hadamard variant stays power-of-two only.
"""

from __future__ import annotations

import math

import numpy as np

MASK64 = (1 << 64) - 1
SPLITMIX_GAMMA = 0x9E3779B97F4A7C15


# --------------------------------------------------------------------------
# Sign vector (reading 1)
# --------------------------------------------------------------------------

def splitmix64(state: int) -> int:
    """The splitmix64 output function applied to a 64-bit state."""
    z = state & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def splitmix64_stream(seed: int, n: int) -> list[int]:
    """First n outputs of a splitmix64 generator seeded with ``seed``.

    The generator adds the golden-ratio increment to its state before each
    output, so output number i is the output function of seed + (i+1)*gamma.
    """
    return [splitmix64((seed + (i + 1) * SPLITMIX_GAMMA) & MASK64) for i in range(n)]


def sign_vector(d: int, seed: int) -> np.ndarray:
    """s in {-1, +1}^d: the fixed random sign vector of the SRFT ([WQF] Methodology 1)."""
    words = splitmix64_stream(seed, d)
    return np.array([-1.0 if (w >> 63) & 1 else 1.0 for w in words], dtype=np.float64)


# --------------------------------------------------------------------------
# SRFT forward / inverse ([WQF] Methodology 1 and 2; readings 2 and 3)
# --------------------------------------------------------------------------

def _check_d(d: int) -> None:
    """The SRFT needs an even d >= 4 (reading 10: [WQF] Methodology 1 credits the SRFT with handling
    dimensions that are not powers of two); the Hadamard variant needs a power of two."""
    if d < 4 or d % 2:
        raise ValueError(f"d must be even and >= 4, got {d}")


def _check_pow2(d: int) -> None:
    if d < 4 or d & (d - 1):
        raise ValueError(f"the Hadamard variant needs a power of two d >= 4, got {d}")


def dft_half_matrix(d: int) -> np.ndarray:
    """Rows k = 0..d/2 of the unitary DFT matrix: F[k, n] = exp(-2 pi i nk/d) / sqrt(d).

    The product nk is reduced mod d before the angle is formed so that the
    cosines and sines are evaluated on small arguments.
    """
    _check_d(d)
    k = np.arange(d // 2 + 1).reshape(-1, 1)
    n = np.arange(d).reshape(1, -1)
    ang = 2.0 * np.pi * ((n * k) % d) / d
    return (np.cos(ang) - 1j * np.sin(ang)) / math.sqrt(d)


def idft_matrix(d: int) -> np.ndarray:
    """The full unitary inverse DFT: G[n, k] = exp(+2 pi i nk/d) / sqrt(d)."""
    _check_d(d)
    n = np.arange(d).reshape(-1, 1)
    k = np.arange(d).reshape(1, -1)
    ang = 2.0 * np.pi * ((n * k) % d) / d
    return (np.cos(ang) + 1j * np.sin(ang)) / math.sqrt(d)


def hermitian_pack(y: np.ndarray) -> np.ndarray:
    """Fold the d/2+1 bins of a real signal's spectrum into d reals (reading 3)."""
    half = y.shape[-1] - 1
    d = 2 * half
    p = np.empty(y.shape[:-1] + (d,), dtype=np.float64)
    p[..., 0] = y[..., 0].real
    p[..., 1] = y[..., half].real
    r2 = math.sqrt(2.0)
    p[..., 2::2] = r2 * y[..., 1:half].real
    p[..., 3::2] = r2 * y[..., 1:half].imag
    return p


def hermitian_unpack(p: np.ndarray) -> np.ndarray:
    """Inverse of ``hermitian_pack``: the full length-d conjugate-symmetric spectrum."""
    d = p.shape[-1]
    half = d // 2
    y = np.zeros(p.shape[:-1] + (d,), dtype=np.complex128)
    y[..., 0] = p[..., 0]
    y[..., half] = p[..., 1]
    r2 = math.sqrt(2.0)
    yk = (p[..., 2::2] + 1j * p[..., 3::2]) / r2
    y[..., 1:half] = yk
    y[..., half + 1 :] = np.conj(yk[..., ::-1])
    return y


def srft_forward(x: np.ndarray, seed: int) -> np.ndarray:
    """p = SRFT(x) = pack(F . diag(s) . x) over the last axis, in fp64."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    u = x * sign_vector(d, seed)
    y = u @ dft_half_matrix(d).T
    return hermitian_pack(y)


def srft_inverse(p: np.ndarray, seed: int) -> np.ndarray:
    """x = diag(s) . F^{-1} . unpack(p): the exact inverse of ``srft_forward``."""
    p = np.asarray(p, dtype=np.float64)
    d = p.shape[-1]
    y = hermitian_unpack(p)
    u = (y @ idft_matrix(d).T).real
    return u * sign_vector(d, seed)


def srft_matrix(d: int, seed: int) -> np.ndarray:
    """R with p = R x, built column by column from ``srft_forward`` of the basis."""
    return srft_forward(np.eye(d), seed).T


# --------------------------------------------------------------------------
# Hadamard variant (reading 8)
# --------------------------------------------------------------------------

def hadamard_matrix(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order d (a power of two), natural order:
    H_ij = (-1)^popcount(i & j)."""
    _check_pow2(d)
    i = np.arange(d)
    parity = np.array([[bin(a & b).count("1") & 1 for b in i] for a in i])
    return np.where(parity == 1, -1.0, 1.0)


def srht_forward(x: np.ndarray, seed: int) -> np.ndarray:
    """SRHT(x) = d^(-1/2) H diag(s) x over the last axis, in fp64."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    return (x * sign_vector(d, seed)) @ hadamard_matrix(d).T / math.sqrt(d)


def srht_inverse(y: np.ndarray, seed: int) -> np.ndarray:
    """x = diag(s) H^T y / sqrt(d), the exact inverse (H H^T = d I)."""
    y = np.asarray(y, dtype=np.float64)
    d = y.shape[-1]
    return (y @ hadamard_matrix(d)) / math.sqrt(d) * sign_vector(d, seed)


def srht_matrix(d: int, seed: int) -> np.ndarray:
    """The SRHT as a d x d matrix, built from ``srht_forward`` of the basis."""
    return srht_forward(np.eye(d), seed).T


TRANSFORMS = ("srft", "srht")


def rotate(x, seed: int, transform: str = "srft") -> np.ndarray:
    """The forward transform named by ``transform``."""
    if transform == "srft":
        return srft_forward(x, seed)
    if transform == "srht":
        return srht_forward(x, seed)
    raise ValueError(f"unknown transform {transform!r}")


def unrotate(p, seed: int, transform: str = "srft") -> np.ndarray:
    """The inverse transform named by ``transform``."""
    if transform == "srft":
        return srft_inverse(p, seed)
    if transform == "srht":
        return srht_inverse(p, seed)
    raise ValueError(f"unknown transform {transform!r}")


# --------------------------------------------------------------------------
# Group quantiser ([WQF] Methodology 2 and 3; readings 4-6)
# --------------------------------------------------------------------------

def qmax(bits: int) -> int:
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    return (1 << (bits - 1)) - 1


SCALE_FORMATS = ("fp32", "fp16", "e8m0")
FP16_MAX = 65504.0


def fp16_round(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest fp16 value (ties to even), saturating at +-65504."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        h = np.clip(v, -FP16_MAX, FP16_MAX).astype(np.float16)
    return h.astype(np.float64)


def e8m0_exponent(v: np.ndarray) -> np.ndarray:
    """ceil(log2(v)) for v > 0, exactly (from the binary exponent and mantissa), clamped to [-126, 127]."""
    v = np.asarray(v, dtype=np.float64)
    m, k = np.frexp(np.where(v > 0, v, 1.0))  # v = m 2^k with m in [0.5, 1)
    e = np.where(m == 0.5, k - 1, k)
    return np.clip(e, -126, 127)


def store_scales(A_over_Q: np.ndarray, scale_format: str):
    """The stored scale (as its fp64 value) and its raw storage (fp32 / fp16 bits / e8m0 bytes), reading 9."""
    if scale_format == "fp32":
        return A_over_Q, A_over_Q.astype(np.float32)
    if scale_format == "fp16":
        v = fp16_round(A_over_Q)
        return v, v.astype(np.float16).view(np.uint16)
    if scale_format == "e8m0":
        e = e8m0_exponent(A_over_Q)
        v = np.where(A_over_Q > 0, np.ldexp(1.0, e), 0.0)
        raw = np.where(A_over_Q > 0, e + 127, 0).astype(np.uint8)
        return v, raw
    raise ValueError(f"unknown scale format {scale_format!r}")


def decode_scales(raw: np.ndarray, scale_format: str) -> np.ndarray:
    """fp64 values of stored scales (the inverse of the raw part of ``store_scales``)."""
    raw = np.asarray(raw)
    if scale_format == "fp32":
        return raw.astype(np.float64)
    if scale_format == "fp16":
        return raw.astype(np.uint16).view(np.float16).astype(np.float64)
    if scale_format == "e8m0":
        b = raw.astype(np.int64)
        return np.where(b > 0, np.ldexp(1.0, b - 127), 0.0)
    raise ValueError(f"unknown scale format {scale_format!r}")


def quantize_groups(z: np.ndarray, bits: int, group: int, scale_format: str = "fp32"):
    """Per-group absmax quantisation of the rotated, rescaled vector z.

    Returns (q, scale, r): the integer codes, the fp64 group scales (A_j / Q,
    or its stored fp16 / e8m0 value, reading 9) and the pre-round values
    r_i = z_i / scale_j (0 where the scale is 0).
    """
    z = np.asarray(z, dtype=np.float64)
    d = z.shape[-1]
    if group <= 0 or d % group:
        raise ValueError("group must divide d")
    Q = qmax(bits)
    zg = z.reshape(z.shape[:-1] + (d // group, group))
    A = np.max(np.abs(zg), axis=-1)
    scale, _ = store_scales(A / Q, scale_format)
    safe = np.where(scale > 0, scale, 1.0)
    r = np.where(scale[..., None] > 0, zg / safe[..., None], 0.0)
    q = np.clip(np.rint(r), -Q, Q).astype(np.int64)
    return q.reshape(z.shape), scale, r.reshape(z.shape)


def pack_codes(q: np.ndarray, bits: int) -> np.ndarray:
    """Bytes of the code plane: int4 two per byte (even index low), int8 one per byte."""
    q = np.asarray(q, dtype=np.int64)
    if bits == 8:
        return (q & 0xFF).astype(np.uint8)
    if bits == 4:
        lo = q[..., 0::2] & 0xF
        hi = q[..., 1::2] & 0xF
        return (lo | (hi << 4)).astype(np.uint8)
    raise ValueError("bits must be 4 or 8")


def unpack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Signed integer codes from the code plane (inverse of ``pack_codes``)."""
    c = np.asarray(codes, dtype=np.int64)
    if bits == 8:
        return np.where(c >= 128, c - 256, c)
    if bits == 4:
        lo = c & 0xF
        hi = (c >> 4) & 0xF
        lo = np.where(lo >= 8, lo - 16, lo)
        hi = np.where(hi >= 8, hi - 16, hi)
        out = np.empty(c.shape[:-1] + (2 * c.shape[-1],), dtype=np.int64)
        out[..., 0::2] = lo
        out[..., 1::2] = hi
        return out
    raise ValueError("bits must be 4 or 8")


# --------------------------------------------------------------------------
# Codec: quantise / dequantise a K or V tensor
# --------------------------------------------------------------------------

def srft_kv_quantize(x, lam, bits: int, group: int, seed: int, transform: str = "srft",
                     scale_format: str = "fp32") -> dict:
    """Encode head vectors x[..., d] (fp16 values, any leading shape).

    lam is None (all ones) or broadcastable to x.  Returns a dict with the
    packed ``codes`` (uint8), fp64 ``scales`` [..., d/group] (the stored
    values), their raw storage ``scales_raw``, the unrounded ``a_over_q``
    (A_j / Q), the integer codes ``q``, the pre-round values ``r`` and the
    rotated, rescaled ``z``.  ``transform`` selects the SRFT (default) or the
    SRHT (reading 8); ``scale_format`` the scale plane (reading 9).
    """
    x = np.asarray(x, dtype=np.float64)
    p = rotate(x, seed, transform)
    z = p if lam is None else p * np.asarray(lam, dtype=np.float64)
    q, scale, r = quantize_groups(z, bits, group, scale_format)
    d = z.shape[-1]
    a_over_q = np.max(np.abs(z.reshape(z.shape[:-1] + (d // group, group))), axis=-1) / qmax(bits)
    return {"codes": pack_codes(q, bits), "scales": scale, "scales_raw": store_scales(a_over_q, scale_format)[1],
            "a_over_q": a_over_q, "q": q, "r": r, "z": z}


def dequantize_rotated(codes, scales, lam, bits: int, group: int) -> np.ndarray:
    """p_hat = (q * scale) / lambda: the dequantised vector in the rotated domain."""
    q = unpack_codes(codes, bits).astype(np.float64)
    sc = np.repeat(np.asarray(scales, dtype=np.float64), group, axis=-1)
    zhat = q * sc
    return zhat if lam is None else zhat / np.asarray(lam, dtype=np.float64)


def srft_kv_dequantize(codes, scales, lam, bits: int, group: int, seed: int, transform: str = "srft") -> np.ndarray:
    """x_hat = T^{-1}((q * scale) / lambda) with T the SRFT (or the SRHT), in fp64."""
    return unrotate(dequantize_rotated(codes, scales, lam, bits, group), seed, transform)


# --------------------------------------------------------------------------
# Decode attention on the dequantised cache ([GEM] Flash Attention section)
# --------------------------------------------------------------------------

def decode_attention(q, k_hat, v_hat, seq_lens=None, sm_scale=None) -> np.ndarray:
    """Plain softmax attention of one query token per (batch, query head).

    q: [B, Hq, d]; k_hat, v_hat: [B, T, Hkv, d] (already dequantised,
    unrotated); query head h reads kv head h // (Hq // Hkv).  Exact
    max-subtracted softmax over tokens t < seq_lens[b].  Returns [B, Hq, d].
    """
    q = np.asarray(q, dtype=np.float64)
    k_hat = np.asarray(k_hat, dtype=np.float64)
    v_hat = np.asarray(v_hat, dtype=np.float64)
    B, Hq, d = q.shape
    T, Hkv = k_hat.shape[1], k_hat.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    rep = Hq // Hkv
    if sm_scale is None or sm_scale <= 0:
        sm_scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, Hq, d), dtype=np.float64)
    for b in range(B):
        L = T if seq_lens is None else int(seq_lens[b])
        if L == 0:
            continue
        for h in range(Hq):
            kv = h // rep
            s = sm_scale * (k_hat[b, :L, kv, :] @ q[b, h])
            w = np.exp(s - s.max())
            out[b, h] = (w @ v_hat[b, :L, kv, :]) / w.sum()
    return out


def dequantize_cache(side: dict, seed: int) -> np.ndarray:
    """Unrotated fp64 cache [B, T, H, d] from one side of a cache description.

    side = {"bits": 4|8, "codes", "scales", "lam" (None or [B|1, H, d]),
    "group", optional "transform" ("srft" when absent)} for a packed side, or
    {"bits": 16, "values": [B, T, H, d]} for a raw fp16 side (no rotation, no
    scales).
    """
    if side["bits"] == 16:
        return np.asarray(side["values"], dtype=np.float64)
    lam = side.get("lam")
    if lam is not None:
        lam = np.asarray(lam, dtype=np.float64)[:, None, :, :]
    return srft_kv_dequantize(side["codes"], side["scales"], lam, side["bits"], side["group"], seed,
                              side.get("transform", "srft"))


def packed_decode_attention(q, k_side: dict, v_side: dict, seed: int, seq_lens=None, sm_scale=None):
    """Decode attention over a packed cache: dequantise both sides, then attend."""
    return decode_attention(q, dequantize_cache(k_side, seed), dequantize_cache(v_side, seed), seq_lens, sm_scale)


# --------------------------------------------------------------------------
# Memory accounting ([GEM] INT8/INT4 section; [KVS] memory calculation)
# --------------------------------------------------------------------------

def kv_bytes(layers: int, kv_heads: int, head_dim: int, seq_len: int, dtype_bytes: float) -> float:
    """KV-cache bytes: 2 x layers x kv_heads x head_dim x seq_len x dtype_bytes."""
    return 2 * layers * kv_heads * head_dim * seq_len * dtype_bytes


SCALE_BYTES = {"fp32": 4, "fp16": 2, "e8m0": 1}


def packed_vector_bytes(d: int, bits: int, group: int, scale_bytes: int = 4) -> int:
    """Bytes of one packed head vector: the code plane plus one scale per group."""
    return d * bits // 8 + (d // group) * scale_bytes


def packed_kv_bytes(layers, kv_heads, d, seq_len, bits_k, bits_v, group, scale_bytes=4) -> int:
    """Bytes of a packed K/V cache with separate code and scale planes."""
    per_token = packed_vector_bytes(d, bits_k, group, scale_bytes) + packed_vector_bytes(d, bits_v, group, scale_bytes)
    return layers * kv_heads * seq_len * per_token
