"""Pins of the paged KV-cache write oracle (CPU only)."""
import numpy as np
import torch

from oracle import cache_write as cw
from oracle import e4m3_table


def _finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    return codes, e4m3_table()[codes].astype(np.float32)


def test_every_finite_code_round_trips():
    codes, vals = _finite_codes()
    got = cw.e4m3_encode(vals)
    # +0 and -0 keep their sign bit; every other value maps back to its own code
    assert (got == codes).all()


def test_matches_torch_cast_where_it_does_not_overflow():
    gen = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(200000, generator=gen) * s for s in (0.01, 1.0, 30.0, 150.0)]).float()
    x = torch.cat([x, torch.rand(20000, generator=gen) * 2 ** -6, torch.linspace(-464, 464, 9281)])
    x = x[x.abs() <= 464]  # beyond, the torch cast returns NaN where the definition saturates
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (cw.e4m3_encode(x.numpy()) == ref).all()


def test_ties_go_to_the_even_mantissa_and_large_values_saturate():
    _, vals = _finite_codes()
    pos = np.sort(vals[vals > 0])
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)
    lo_code, hi_code = cw.e4m3_encode(pos[:-1]), cw.e4m3_encode(pos[1:])
    got = cw.e4m3_encode(mids)
    # the even code of the two neighbours (their mantissa's last bit is the code's last bit)
    want = np.where(lo_code % 2 == 0, lo_code, hi_code)
    assert (got == want).all()
    assert (cw.e4m3_encode(np.array([448.0, 480.0, 1e6, np.inf], np.float32)) == 0x7E).all()
    assert (cw.e4m3_encode(np.array([-500.0, -np.inf], np.float32)) == 0xFE).all()
    assert cw.e4m3_encode(np.array([2.0 ** -10], np.float32))[0] == 0x00  # half of 2^-9: even
    assert cw.e4m3_encode(np.array([3 * 2.0 ** -10], np.float32))[0] == 0x02  # 1.5 x 2^-9: even


def test_scatter_puts_new_tokens_at_the_end_of_each_sequence():
    rng = np.random.default_rng(5)
    P, Hkv, NB = 16, 2, 40
    seqs = [(3, 20), (1, 1), (16, 33), (0, 7)]          # (q_len, L)
    perm = rng.permutation(NB)
    bt = np.full((len(seqs), 4), -1, np.int32)
    used = 0
    for s, (q, L) in enumerate(seqs):
        n = (L + P - 1) // P
        bt[s, :n] = perm[used:used + n]
        used += n
    qsl = np.concatenate([[0], np.cumsum([q for q, _ in seqs])]).astype(np.int32)
    sl = np.array([L for _, L in seqs], np.int32)
    T = int(qsl[-1])
    kn = rng.standard_normal((T, Hkv, 256)).astype(np.float32)
    vn = rng.standard_normal((T, Hkv, 256)).astype(np.float32)
    kc0 = rng.integers(0, 256, (NB, P, Hkv, 256)).astype(np.uint8)
    vc0 = rng.integers(0, 256, (NB, P, Hkv, 256)).astype(np.uint8)
    kc, vc = cw.cache_write(kn, vn, kc0, vc0, bt, sl, qsl, 0.5, 2.0)
    written = np.zeros((NB, P), bool)
    for s, (q, L) in enumerate(seqs):
        for t in range(q):
            pos = L - q + t                           # the definition, one token at a time
            page, slot = bt[s, pos // P], pos % P
            written[page, slot] = True
            assert (kc[page, slot] == cw.e4m3_encode(kn[qsl[s] + t] * np.float32(2.0))).all()
            assert (vc[page, slot] == cw.e4m3_encode(vn[qsl[s] + t] * np.float32(0.5))).all()
    assert (kc[~written] == kc0[~written]).all() and (vc[~written] == vc0[~written]).all()
    assert written.sum() == T


def _bf16_values():
    """Every finite non-negative bf16 value, as float32."""
    return (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)


def test_code_is_the_product_with_the_fp32_reciprocal_not_the_division():
    # The reading of the write: code = e4m3(value * fl32(1 / descale)), the product in fp32.
    # For a descale that is not a power of two, a few bf16 inputs sit where value / descale
    # and value * fl32(1 / descale) fall on the two sides of an e4m3 tie; the write must
    # take the product's code there.
    x = _bf16_values()
    d = np.float32(1.7)
    inv = np.float32(1.0) / d
    with np.errstate(over="ignore"):
        by_div, by_mul = cw.e4m3_encode(x / d), cw.e4m3_encode(x * inv)
    differ = np.nonzero(by_div != by_mul)[0]
    assert len(differ) >= 1
    v = float(x[differ[0]])
    P, Hkv = 16, 1
    kn = np.full((1, Hkv, 256), v, np.float32)
    kc0 = np.zeros((2, P, Hkv, 256), np.uint8)
    bt = np.array([[1]], np.int32)
    kc, vc = cw.cache_write(kn, -kn, kc0, kc0, bt, np.array([5], np.int32), np.array([0, 1], np.int32),
                            float(d), float(d))
    assert (kc[1, 4] == by_mul[differ[0]]).all() and (kc[1, 4] != by_div[differ[0]]).all()
    assert (vc[1, 4] == (by_mul[differ[0]] | 0x80)).all()
