"""Pins of the quantized-KV oracle (int8 and fp8 E4M3 codes, one fp32 scale
per (token, kv head) row) against things other than itself.

The pages name an 8-bit KV cache as the lever that halves each decode's read
("Contiguous vs Paged KV Cache on RDNA4", section "The order of the memory
levers") but fix no format; the oracle's reading is stated in its C header.

- The E4M3 codec is checked against torch's float8_e4m3fn conversion (a
  library routine) on every code and on exact values, midpoints and random
  values up to 464; saturation above that follows the format's definition.
- Quantized rows are recomputed with torch fp32 ops (division, round half to
  even, float8 conversion), independently of the oracle's C code.
- Dequantization error bounds follow from the formats.
- The quantized decode equals torch's scaled_dot_product_attention in fp64 on
  K/V that the test dequantizes itself.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle

KINDS = ["int8", "fp8_e4m3"]
QMAX = {"int8": 127.0, "fp8_e4m3": 448.0}


def _lib_decode(codes: torch.Tensor) -> torch.Tensor:
    return codes.view(torch.float8_e4m3fn).to(torch.float64)


def test_e4m3_decode_matches_library_on_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = _lib_decode(codes)
    ours = torch.tensor([oracle.e4m3_decode(c) for c in range(256)], dtype=torch.float64)
    nan = torch.isnan(ref)
    assert torch.equal(nan, torch.isnan(ours)) and int(nan.sum()) == 2   # S.1111.111
    assert torch.equal(ref[~nan], ours[~nan])
    # landmarks of the format: smallest subnormal, largest subnormal, smallest
    # normal, one, largest finite
    assert ours[0x01] == 2.0 ** -9 and ours[0x07] == 7 * 2.0 ** -9
    assert ours[0x08] == 2.0 ** -6 and ours[0x38] == 1.0 and ours[0x7E] == 448.0
    assert torch.all(ours[1:0x7F] > ours[0:0x7E])                       # increasing


def _finite_values():
    v = np.array([oracle.e4m3_decode(c) for c in range(0x7F)], dtype=np.float64)
    return v   # 0 .. 448, increasing


def test_e4m3_encode_matches_library():
    v = _finite_values()
    mids = (v[1:] + v[:-1]) / 2                     # exact ties (all fit in fp32)
    g = torch.Generator().manual_seed(5)
    mag = torch.exp2(torch.empty(20000, dtype=torch.float64).uniform_(-12, math.log2(464),
                                                                      generator=g))
    rnd = mag.numpy() * np.where(torch.rand(20000, generator=g).numpy() < 0.5, -1, 1)
    xs = np.concatenate([v, -v, mids, -mids, rnd, [463.99, 464.0, -464.0]]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    bad = np.nonzero(ref != ours)[0]
    assert bad.size == 0, [(float(xs[i]), int(ref[i]), int(ours[i])) for i in bad[:5]]


def test_e4m3_encode_saturates_above_464():
    for x in (464.0001, 470.0, 480.0, 1e6, 3e38, float("inf")):
        assert oracle.e4m3_encode(x) == 0x7E and oracle.e4m3_encode(-x) == 0xFE


def _rows(act, n, D, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, D, generator=g) * std).to(act)


def _expected_row(kind, x):
    """Codes and scale of one row, recomputed with torch fp32 ops."""
    xf = x.to(torch.float32)
    a = xf.abs().max()
    s = (a / torch.tensor(QMAX[kind], dtype=torch.float32)).to(torch.float32)
    if float(a) == 0.0:
        return torch.zeros(x.shape[0], dtype=torch.uint8), s
    v = xf / s
    if kind == "int8":
        c = torch.round(v).clamp(-127, 127).to(torch.int8).view(torch.uint8)
    else:
        c = v.to(torch.float8_e4m3fn).view(torch.uint8)
    return c, s


def _quantize_rows(kind, rows):
    """Quantize rows [n][D] through the oracle's append (one slot per row)."""
    n, D = rows.shape
    kc = torch.zeros(n, 1, 1, D, dtype=torch.uint8)
    vc = torch.zeros_like(kc)
    ks = torch.zeros(n, 1, 1, dtype=torch.float32)
    vs = torch.zeros_like(ks)
    kn = rows.reshape(n, 1, D)
    oracle.append_quant(kind, kn, kn.clone(), torch.arange(n), kc, vc, ks, vs)
    assert torch.equal(kc, vc) and torch.equal(ks, vs)
    return kc.reshape(n, D), ks.reshape(n)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("act", [torch.float16, torch.bfloat16])
def test_quantized_rows_match_torch(kind, act):
    rows = torch.cat([_rows(act, 60, 128, 11), _rows(act, 4, 128, 12, std=1e-4),
                      _rows(act, 4, 128, 13, std=300.0)])
    codes, scales = _quantize_rows(kind, rows)
    for i in range(rows.shape[0]):
        c, s = _expected_row(kind, rows[i])
        assert torch.equal(codes[i], c), f"row {i}"
        assert scales[i].item() == s.item(), f"row {i}"


def test_int8_ties_round_to_even_and_extremes():
    # max |x| = 127 makes the scale exactly 1, so x / s = x: exact ties
    row = torch.tensor([127.0, 0.5, 1.5, 2.5, -0.5, -2.5, 126.5, -127.0], dtype=torch.bfloat16)
    codes, scales = _quantize_rows("int8", row.reshape(1, -1))
    assert scales[0].item() == 1.0
    assert codes[0].view(torch.int8).tolist() == [127, 0, 2, 2, 0, -2, 126, -127]


def test_e4m3_ties_round_to_even():
    # max |x| = 448 makes the scale exactly 1; midpoints between E4M3 values
    v = _finite_values()
    mids = ((v[1:] + v[:-1]) / 2)[::9][:20]
    row = torch.tensor(np.concatenate([[448.0], mids]), dtype=torch.float32).to(torch.float16)
    assert torch.equal(row.to(torch.float64), torch.from_numpy(np.concatenate([[448.0], mids])))
    codes, scales = _quantize_rows("fp8_e4m3", row.reshape(1, -1))
    assert scales[0].item() == 1.0
    ours = codes[0].tolist()
    for m, c in zip(mids, ours[1:]):
        lo = int(np.searchsorted(v, m)) - 1          # the neighbours are lo and lo + 1
        assert c in (lo, lo + 1) and c % 2 == 0, (m, c)


@pytest.mark.parametrize("kind", KINDS)
def test_zero_row_has_zero_scale_and_codes(kind):
    codes, scales = _quantize_rows(kind, torch.zeros(1, 64, dtype=torch.float16))
    assert scales[0].item() == 0.0 and int(codes.sum()) == 0


def _dequant(kind, codes, scales):
    if kind == "int8":
        val = codes.view(torch.int8).to(torch.float64)
    else:
        val = _lib_decode(codes)
    return val * scales.to(torch.float64).unsqueeze(-1)


@pytest.mark.parametrize("kind", KINDS)
def test_dequantization_error_bounds(kind):
    rows = _rows(torch.bfloat16, 200, 128, 21)
    codes, scales = _quantize_rows(kind, rows)
    x = rows.to(torch.float64)
    xh = _dequant(kind, codes, scales)
    s = scales.to(torch.float64).unsqueeze(-1)
    err = (x - xh).abs()
    if kind == "int8":
        # half a step, plus the fp32 rounding of x / s
        assert torch.all(err <= s * (0.5 + 1e-5))
    else:
        # normal range: half an ulp of a 3-bit mantissa, relative to |x / s|
        # (slack for the fp32 division); subnormal range: half of 2^-9
        v = (x / s).abs()
        ulp = torch.where(v >= 2.0 ** -6, torch.exp2(torch.floor(torch.log2(v)) - 3),
                          torch.full_like(v, 2.0 ** -9))
        assert torch.all(err <= s * (0.5 * ulp + 1e-5 * v + 1e-12))
    # the largest element of each row is reproduced to the top code
    top = x.abs().argmax(dim=1)
    q = codes.view(torch.int8) if kind == "int8" else codes
    tops = q[torch.arange(200), top]
    if kind == "int8":
        assert torch.all(tops.abs() == 127)
    else:
        assert torch.all((tops & 0x7F) == 0x7E)


def _paged_case(kind, act, S, Hq, Hk, D, B, lens, seed):
    """Random activations for every token, quantized into a shuffled pool by
    the oracle's append; returns the pieces and the contiguous activations."""
    g = torch.Generator().manual_seed(seed)
    nblk = [(L + B - 1) // B for L in lens]
    NB = sum(nblk) + 3
    perm = torch.randperm(NB, generator=g)
    M = max(max(nblk), 1)
    tables = torch.full((S, M), -1, dtype=torch.int32)
    k = 0
    slots = []
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[k:k + n].to(torch.int32)
        k += n
        for t in range(lens[s]):
            slots.append(int(tables[s, t // B]) * B + t % B)
    T = len(slots)
    kn = torch.randn(T, Hk, D, generator=g).to(act)
    vn = torch.randn(T, Hk, D, generator=g).to(act)
    q = torch.randn(S, Hq, D, generator=g).to(act)
    kc = torch.full((NB, Hk, B, D), 0x7F, dtype=torch.uint8)   # NaN / 127 sentinels
    vc = kc.clone()
    ks = torch.full((NB, Hk, B), float("nan"), dtype=torch.float32)
    vs = ks.clone()
    oracle.append_quant(kind, kn, vn, torch.tensor(slots, dtype=torch.int64), kc, vc, ks, vs)
    return q, kc, vc, ks, vs, tables, torch.tensor(lens, dtype=torch.int32)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("act,Hq,Hk,B", [(torch.bfloat16, 8, 2, 16), (torch.float16, 4, 4, 8),
                                         (torch.bfloat16, 6, 2, 32)])
def test_decode_quant_equals_sdpa_on_dequantized_cache(kind, act, Hq, Hk, B):
    S, D = 3, 64
    lens = [1, 37, 70]
    q, kc, vc, ks, vs, tables, cl = _paged_case(kind, act, S, Hq, Hk, D, B, lens, seed=31)
    scale = 1.0 / math.sqrt(D)
    got = oracle.decode_quant(kind, q, kc, vc, ks, vs, tables, cl, scale)
    kd, vd = _dequant(kind, kc, ks), _dequant(kind, vc, vs)
    G = Hq // Hk
    for s in range(S):
        L = lens[s]
        idx = [int(tables[s, t // B]) for t in range(L)]
        off = [t % B for t in range(L)]
        K = torch.stack([kd[idx[t], :, off[t]] for t in range(L)], dim=1)   # [Hk][L][D]
        V = torch.stack([vd[idx[t], :, off[t]] for t in range(L)], dim=1)
        Kq = K.repeat_interleave(G, dim=0)
        Vq = V.repeat_interleave(G, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[s].to(torch.float64).unsqueeze(1), Kq, Vq, scale=scale).squeeze(1)
        assert np.max(np.abs(got[s] - ref.numpy())) < 1e-12


@pytest.mark.parametrize("kind", KINDS)
def test_append_quant_writes_only_its_slots(kind):
    NB, Hk, B, D = 6, 2, 16, 64
    kc = torch.full((NB, Hk, B, D), 0xA5, dtype=torch.uint8)
    vc = kc.clone()
    ks = torch.full((NB, Hk, B), -7.0)
    vs = ks.clone()
    g = torch.Generator().manual_seed(41)
    kn = torch.randn(3, Hk, D, generator=g).to(torch.float16)
    vn = torch.randn(3, Hk, D, generator=g).to(torch.float16)
    slots = torch.tensor([5 * B + 3, -1, 0], dtype=torch.int64)
    oracle.append_quant(kind, kn, vn, slots, kc, vc, ks, vs)
    touched = torch.zeros(NB, Hk, B, dtype=torch.bool)
    touched[5, :, 3] = True
    touched[0, :, 0] = True
    assert torch.all(kc[~touched] == 0xA5) and torch.all(vc[~touched] == 0xA5)
    assert torch.all(ks[~touched] == -7.0) and torch.all(vs[~touched] == -7.0)
    for blk, off, i in ((5, 3, 0), (0, 0, 2)):
        for g_ in range(Hk):
            c, s = _expected_row(kind, kn[i, g_])
            assert torch.equal(kc[blk, g_, off], c) and ks[blk, g_, off].item() == s.item()
            c, s = _expected_row(kind, vn[i, g_])
            assert torch.equal(vc[blk, g_, off], c) and vs[blk, g_, off].item() == s.item()
    with pytest.raises(ValueError):
        oracle.append_quant(kind, kn, vn, torch.tensor([NB * B, 0, 0]), kc, vc, ks, vs)
