"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test names what it pins: a hand-worked example, a closed form, an
independent library routine (numpy's IEEE fp16 conversion, exact rational
arithmetic) or an invariant that a plausible slip (dropped term, wrong sign,
wrong index, swapped operands) would break.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as O
from kv_cache_compression_decode_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _table(d):
    f = np.zeros(256, dtype=np.uint32)
    for k, v in d.items():
        f[int(k)] = v
    return f


# --------------------------------------------------------------------------
# fp16 <-> fp32 against numpy's independent IEEE implementation
# --------------------------------------------------------------------------

def test_f16_to_f32_all_halves_match_numpy():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_round_to_nearest_even_matches_numpy():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=400_000, dtype=np.uint64).astype(np.uint32)
    # dense coverage of the half range, ties and subnormal boundaries
    edges = []
    for h in range(0, 0x7C01):
        f = np.uint16(h).view(np.float16).astype(np.float32).view(np.uint32)
        edges += [int(f) - 1, int(f), int(f) + 1, int(f) + 0x1000, int(f) + 0xFFF, int(f) + 0x1001]
    edges = np.array([e & 0xFFFFFFFF for e in edges], dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([bits, edges, edges | np.uint32(0x80000000)])
    f = bits.view(np.float32)
    ours = O.f32_to_f16(f)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(np.isnan(ours.view(np.float16)), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# --------------------------------------------------------------------------
# layer bins and group geometry
# --------------------------------------------------------------------------

def test_layer_steps_follow_layer_thirds():
    # shallow / middle / deep thirds get 0.5 / 1.0 / 1.5
    s32 = O.layer_steps(32)
    assert list(s32[:11]) == [0.5] * 11 and list(s32[11:22]) == [1.0] * 11 and list(s32[22:]) == [1.5] * 10
    assert list(O.layer_steps(4)) == [0.5, 0.5, 1.0, 1.5]
    s80 = O.layer_steps(80)
    assert [int((s80 == v).sum()) for v in (0.5, 1.0, 1.5)] == [27, 27, 26]  # l<27, 27<=l<54, l>=54
    assert list(O.layer_steps(3, mult=4.0)) == [2.0, 4.0, 6.0]


@pytest.mark.parametrize("T,chunk,G,A", [(256, 256, 10, 26), (16384, 1536, 10, 10 * 154 + 103),
                                         (16384, 16384, 10, 1639), (7, 3, 2, 5), (5, 5, 1, 5)])
def test_anchor_rows_restart_at_chunks(T, chunk, G, A):
    cfg = O.Config(1, T, 32, G, chunk, chunk, O.layer_steps(1))
    m = O.anchor_mask(cfg)
    expect = np.array([(t % chunk) % G == 0 for t in range(T)])
    assert np.array_equal(m, expect)
    assert O.geometry(cfg)["A"] == A == int(expect.sum())


# --------------------------------------------------------------------------
# table normalization: hand-worked cases and invariants
# --------------------------------------------------------------------------

def test_normalize_hand_examples():
    for ex in json.load(open(os.path.join(GOLD, "normalize_hand_examples.json")))["examples"]:
        f, lo, hi = O.normalize(_table(ex["counts"]))
        assert (lo, hi) == (ex["lo"], ex["hi"]), ex["name"]
        assert np.array_equal(f, _table(ex["freq"])), ex["name"]


def test_normalize_invariants_random():
    rng = np.random.default_rng(7)
    for it in range(300):
        n = np.zeros(256, dtype=np.uint32)
        W = int(rng.integers(1, 257))
        lo = int(rng.integers(0, 257 - W))
        kind = it % 3
        if kind == 0:
            vals = rng.integers(0, 1000, W)
        elif kind == 1:
            vals = (rng.pareto(0.7, W) * 10).astype(np.int64)
        else:
            vals = rng.integers(0, 2, W) * rng.integers(1, 10**6, W)
        n[lo:lo + W] = vals
        if n.sum() == 0:
            n[lo] = 1
        f, flo, fhi = O.normalize(n)
        nz = np.nonzero(n)[0]
        assert (flo, fhi) == (nz.min(), nz.max())
        assert int(f.sum()) == 65536
        assert (f[flo:fhi + 1] >= 1).all() and f[:flo].sum() == 0 and f[fhi + 1:].sum() == 0
        # every f sits near its exact share; the correction moves at most W slots
        N = int(n.sum())
        exact = n[flo:fhi + 1].astype(np.float64) * 65536 / N
        assert np.abs(f[flo:fhi + 1] - exact).max() <= (fhi - flo + 2) + 1


def test_normalize_cross_entropy_close_to_entropy():
    # with large counts the 16-bit table costs almost nothing over the counts
    rng = np.random.default_rng(3)
    q = np.clip(np.rint(rng.normal(0, 2.0, 200_000)), -127, 127).astype(np.int64) + 127
    n = np.bincount(q, minlength=256).astype(np.uint32)
    f, lo, hi = O.normalize(n)
    p = n / n.sum()
    m = n > 0
    H = -(p[m] * np.log2(p[m])).sum()
    X = -(p[m] * np.log2(f[m] / 65536.0)).sum()
    assert H <= X <= H + 1e-3


# --------------------------------------------------------------------------
# range coder
# --------------------------------------------------------------------------

def test_rans_hand_examples():
    for ex in json.load(open(os.path.join(GOLD, "rans_hand_examples.json")))["examples"]:
        freq = np.stack([_table(d) for d in ex["freq"]])
        sym = np.array(ex["symbols"], dtype=np.uint8)
        words = O.rans_encode(sym, freq)
        assert list(words) == ex["words"], ex["name"]
        dec, used = O.rans_decode(words, sym.shape[0], freq)
        assert np.array_equal(dec, sym) and used == len(words), ex["name"]


@pytest.mark.parametrize("lanes", [1, 5, 32])
def test_rans_uniform_power_of_two_table_word_count(lanes):
    # 16 symbols of frequency 4096 are 4 bits each: a lane holding 17 + 4k bits
    # renormalizes before its 4th, 8th, ... symbol (counted from the end), so a
    # stream of n steps is lanes * (2 + floor(n / 4)) words.
    freq = np.zeros((lanes, 256), dtype=np.uint32)
    freq[:, 100:116] = 4096
    rng = np.random.default_rng(lanes)
    for n in range(1, 41):
        sym = rng.integers(100, 116, (n, lanes)).astype(np.uint8)
        w = O.rans_encode(sym, freq)
        assert len(w) == lanes * (2 + n // 4)
        dec, used = O.rans_decode(w, n, freq)
        assert np.array_equal(dec, sym) and used == len(w)


def test_rans_single_symbol_table_costs_only_the_flush():
    lanes, steps = 32, 500
    freq = np.zeros((lanes, 256), dtype=np.uint32)
    freq[np.arange(lanes), np.arange(lanes) + 90] = 65536
    sym = np.tile((np.arange(lanes) + 90).astype(np.uint8), (steps, 1))
    w = O.rans_encode(sym, freq)
    assert list(w) == [1, 0] * lanes  # every state stays at 2^16
    dec, _ = O.rans_decode(w, steps, freq)
    assert np.array_equal(dec, sym)


def _ideal_bits(sym, freq):
    """-log2 of the exact arithmetic-coding interval, per lane (Fractions)."""
    out = []
    for i in range(sym.shape[1]):
        width = Fraction(1)
        for s in sym[:, i]:
            width *= Fraction(int(freq[i, s]), 65536)
        out.append(-math.log2(width.numerator) + math.log2(width.denominator))
    return out


def test_rans_length_against_exact_arithmetic_coding():
    rng = np.random.default_rng(11)
    for it in range(60):
        lanes = int(rng.integers(1, 33))
        steps = int(rng.integers(1, 65))
        freq = np.zeros((lanes, 256), dtype=np.uint32)
        for i in range(lanes):
            W = int(rng.integers(1, 12))
            lo = int(rng.integers(0, 256 - W))
            cnt = np.zeros(256, dtype=np.uint32)
            cnt[lo:lo + W] = rng.integers(1, 50, W)
            freq[i], _, _ = O.normalize(cnt)
        sym = np.zeros((steps, lanes), dtype=np.uint8)
        for i in range(lanes):
            nz = np.nonzero(freq[i])[0]
            p = freq[i, nz] / 65536.0
            sym[:, i] = rng.choice(nz, size=steps, p=p / p.sum())
        w = O.rans_encode(sym, freq)
        ideal = sum(_ideal_bits(sym, freq))
        body = 16 * (len(w) - 2 * lanes)  # words minus the 32-bit flush per lane
        # never more than 2 bytes per lane over the exact interval, never
        # below it by more than the 16 bits the initial state carries
        assert body <= ideal + 16 * lanes + 1e-9
        assert 16 * len(w) >= ideal - 16 * lanes - 1e-9
        dec, used = O.rans_decode(w, steps, freq)
        assert np.array_equal(dec, sym) and used == len(w)


def test_rans_decode_flags_corruption():
    rng = np.random.default_rng(5)
    lanes, steps = 32, 200
    cnt = np.zeros(256, dtype=np.uint32)
    cnt[120:135] = rng.integers(1, 100, 15)
    f, _, _ = O.normalize(cnt)
    freq = np.tile(f, (lanes, 1))
    nz = np.nonzero(f)[0]
    sym = rng.choice(nz, size=(steps, lanes)).astype(np.uint8)
    w = O.rans_encode(sym, freq)
    with pytest.raises(O.OracleError) as e:
        O.rans_decode(w[:-1], steps, freq)  # truncated
    assert e.value.code == O.ERR_CORRUPT
    bad = w.copy()
    bad[3] ^= 0x0100  # initial state of lane 1
    with pytest.raises(O.OracleError) as e:
        O.rans_decode(bad, steps, freq)
    assert e.value.code == O.ERR_CORRUPT
    # a trailing word is left unconsumed; the stream framing (padding check) rejects it
    _, used = O.rans_decode(np.concatenate([w, np.zeros(1, np.uint16)]), steps, freq)
    assert used == len(w)


# --------------------------------------------------------------------------
# quantization: closed form, error bound, special cases
# --------------------------------------------------------------------------

def _closed_form_cache(L, T, C, G, chunk, steps, rng):
    """Anchors on a 0.25 grid with absmax 127/4 per channel (so s = 0.25
    exactly) and every other token = its anchor + k * step for integer k."""
    cfg = O.Config(L, T, C, G, chunk, chunk, np.asarray(steps, np.float32))
    am = O.anchor_mask(cfg)
    a = rng.integers(-127, 128, (L, 2, T, C))
    a[:, :, np.nonzero(am)[0][0], :] = 127  # absmax 127 on the first anchor row
    k = rng.integers(-40, 41, (L, 2, T, C))
    x = np.zeros((L, 2, T, C))
    last = None
    for t in range(T):
        if am[t]:
            last = a[:, :, t, :] * 0.25
            x[:, :, t, :] = last
            k[:, :, t, :] = 0
        else:
            x[:, :, t, :] = last + k[:, :, t, :] * np.asarray(steps)[:, None, None]
    return cfg, x.astype(np.float16), a, k, am


def test_quantize_closed_form_delta_against_group_anchor():
    rng = np.random.default_rng(2)
    steps = [0.5, 1.0, 1.5]
    cfg, x, a, k, am = _closed_form_cache(3, 47, 64, 10, 20, steps, rng)
    scales = O.anchor_scales(cfg, x)
    assert np.all(scales == np.float32(0.25))
    anchors, q = O.quantize(cfg, x, scales)
    assert np.array_equal(anchors, a[:, :, am, :].astype(np.int8))
    assert np.array_equal(q, k)  # delta vs the group's anchor, divided by the layer's step
    enc = O.encode(cfg, x)
    y = O.decode(cfg, enc)
    assert np.array_equal(y, x.view(np.uint16))  # exact grid: lossless


# Hand-worked rounding cases (tests/golden/quantize_hand_examples.{json,txt}).
# They fix what the closed-form grid cannot: ties are rounded to even, not
# away from zero, and the quantizers multiply by the rounded inverse of the
# scale / step instead of dividing by it.

def _quant_examples():
    return json.load(open(os.path.join(GOLD, "quantize_hand_examples.json")))["examples"]


def _rn32(v: Fraction) -> Fraction:
    """Nearest binary32 value to the rational v (normal range), ties to even."""
    if v == 0:
        return Fraction(0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    n = math.floor(a / ulp)
    r = a / ulp - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return (n * ulp) if v > 0 else -(n * ulp)


def _round_int(v: Fraction, half_even: bool) -> int:
    n = math.floor(v)
    r = v - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and (n % 2 == 1 if half_even else v > 0)):
        n += 1
    return n


def _derive(ex, reading):
    """(anchors, q) of an example by exact rational arithmetic under a reading:
    'r' = the codec's (multiply by RN(1/s), ties to even), 'round_half_away',
    'true_division'."""
    vals = [Fraction(float.fromhex(v)) for v in ex["values"]]
    G, step = ex["G"], Fraction(ex["step"])
    half_even = reading != "round_half_away"
    s = _rn32(max(abs(v) for i, v in enumerate(vals) if i % G == 0) / 127)
    r_a, r = _rn32(1 / s), _rn32(1 / step)
    anchors, q, xa = [], [], None
    for i, v in enumerate(vals):
        if i % G == 0:
            t = _rn32(v / s) if reading == "true_division" else _rn32(v * r_a)
            qa = max(-127, min(127, _round_int(t, half_even)))
            anchors.append(qa)
            xa = _rn32(qa * s)
            q.append(None)
        else:
            d = _rn32(v - xa)
            t = _rn32(d / step) if reading == "true_division" else _rn32(d * r)
            q.append(_round_int(t, half_even))
    return s, anchors, q


@pytest.mark.parametrize("ex", _quant_examples(), ids=lambda e: e["name"][:40])
def test_quantize_hand_examples_derivation(ex):
    # the stored values follow the reading, and every other reading listed
    # gives different codes, so each case catches that slip
    s, anchors, q = _derive(ex, "r")
    assert np.float32(float(s)).view(np.uint32) == int(ex["scale_bits"], 16)
    assert anchors == ex["anchors"] and q == ex["q"]
    for name, alt in ex["other_readings"].items():
        _, a2, q2 = _derive(ex, name)
        assert a2 == alt["anchors"] and q2 == alt.get("q", q2)
        assert (a2, q2) != (anchors, q), name


@pytest.mark.parametrize("ex", _quant_examples(), ids=lambda e: e["name"][:40])
def test_quantize_hand_examples(ex):
    vals = np.array([float.fromhex(v) for v in ex["values"]], dtype=np.float16)
    assert vals.astype(np.float64).tolist() == ex["decimal"]  # exact fp16 inputs
    T, G = len(vals), ex["G"]
    cfg = O.Config(1, T, 32, G, T, T, np.array([ex["step"]], np.float32))
    x = np.zeros((1, 2, T, 32), dtype=np.float16)
    x[0, :, :, 0] = vals
    scales = O.anchor_scales(cfg, x)
    assert scales[0, :, 0].view(np.uint32).tolist() == [int(ex["scale_bits"], 16)] * 2
    anchors, q = O.quantize(cfg, x, scales)
    am = O.anchor_mask(cfg)
    for kv in range(2):
        assert anchors[0, kv, :, 0].tolist() == ex["anchors"]
        assert q[0, kv, ~am, 0].tolist() == [v for v in ex["q"] if v is not None]
    y = O.decode(cfg, O.encode(cfg, x))
    expect = np.array(ex["recon"], dtype=np.float16).view(np.uint16)
    assert np.array_equal(y[0, 0, :, 0], expect) and np.array_equal(y[0, 1, :, 0], expect)


def _bound_check(cfg, x, y, scales):
    am = O.anchor_mask(cfg)
    xf = x.astype(np.float64)
    yf = y.view(np.float16).astype(np.float64)
    err = np.abs(xf - yf)
    ulp16 = np.spacing(np.abs(yf).astype(np.float16)).astype(np.float64)
    mag = np.maximum(np.abs(xf), np.abs(yf))
    ulp32 = np.spacing(mag.astype(np.float32)).astype(np.float64)
    steps = np.asarray(cfg.step, np.float64)[:, None, None, None]
    s = scales.astype(np.float64)[:, :, None, :]
    bound_d = steps / 2 + 4 * ulp32 + ulp16 / 2
    bound_a = s / 2 + 4 * ulp32 + ulp16 / 2
    assert (err[:, :, ~am, :] <= np.broadcast_to(bound_d, err.shape)[:, :, ~am, :]).all()
    assert (err[:, :, am, :] <= np.broadcast_to(bound_a, err.shape)[:, :, am, :]).all()


def test_reconstruction_error_bound_synthetic():
    w = synth.small("t", 3, 300, 96, seed=4, rho=0.9, n_outlier=1)
    x = w.generate().numpy()
    cfg = O.Config(3, 300, 96, 10, 128, 64, O.layer_steps(3))
    enc = O.encode(cfg, x)
    y = O.decode(cfg, enc)
    _bound_check(cfg, x, y, enc.scales)


def test_huge_step_gives_all_zero_deltas():
    w = synth.small("t", 2, 64, 32, seed=9)
    x = w.generate().numpy()
    cfg = O.Config(2, 64, 32, 10, 64, 64, np.array([1e6, 1e6], np.float32))
    sc = O.anchor_scales(cfg, x)
    anchors, q = O.quantize(cfg, x, sc)
    assert not q.any()
    y = O.decode(cfg, O.encode(cfg, x))
    am = O.anchor_mask(cfg)
    idx = np.maximum.accumulate(np.where(am, np.arange(64), 0))
    assert np.array_equal(y, y[:, :, idx, :])  # every token equals its anchor


def test_constant_and_zero_channels():
    x = np.zeros((1, 2, 25, 64), dtype=np.float16)
    x[0, 0, :, 1] = 3.0
    x[0, 1, :, 2] = -0.125
    cfg = O.Config(1, 25, 64, 10, 25, 25, np.array([0.5], np.float32))
    sc = O.anchor_scales(cfg, x)
    assert sc[0, 0, 0] == 1.0 and sc[0, 0, 1] == np.float32(3.0) / np.float32(127.0)
    anchors, q = O.quantize(cfg, x, sc)
    assert anchors[0, 0, :, 1].tolist() == [127] * 3 and anchors[0, 1, :, 2].tolist() == [-127] * 3
    y = O.decode(cfg, O.encode(cfg, x))
    assert np.array_equal(y, x.view(np.uint16))


def test_escapes_round_trip_in_step_lane_order():
    T, C = 23, 64
    x = np.zeros((1, 2, T, C), dtype=np.float16)
    x[0, 0, 1, 3] = 200.0   # q = 400 with step 0.5 -> escape
    x[0, 0, 2, 1] = -90.0   # q = -180 -> escape, earlier lane, later step
    x[0, 0, 2, 40] = 64.0   # q = 128 -> escape, second stream group
    x[0, 1, 5, 0] = 63.5    # q = 127 -> largest in-alphabet symbol
    cfg = O.Config(1, T, C, 10, T, T, np.array([0.5], np.float32))
    enc = O.encode(cfg, x)
    assert enc.escapes.tolist() == [400, -180, 128]
    assert enc.esc_off.tolist() == [0, 2, 3, 3, 3]
    y = O.decode(cfg, enc)
    assert np.array_equal(y, x.view(np.uint16))


def test_group_size_one_has_no_deltas_and_empty_streams():
    w = synth.small("t", 1, 40, 64, seed=1)
    x = w.generate().numpy()
    cfg = O.Config(1, 40, 64, 1, 40, 16, O.layer_steps(1))
    enc = O.encode(cfg, x)
    assert enc.payload.size == 0 and enc.escapes.size == 0
    assert (enc.tables.reshape(-1, 2) == [1, 0]).all()  # every table empty
    y = O.decode(cfg, enc)
    _bound_check(cfg, x, y, enc.scales)


def test_single_token():
    x = np.full((2, 2, 1, 32), 1.5, dtype=np.float16)
    cfg = O.Config(2, 1, 32, 10, 1, 1, O.layer_steps(2))
    enc = O.encode(cfg, x)
    assert enc.payload.size == 0
    assert np.array_equal(O.decode(cfg, enc), x.view(np.uint16))


def test_nonfinite_and_invalid_arguments():
    x = np.zeros((1, 2, 30, 32), dtype=np.float16)
    x[0, 1, 17, 5] = np.inf
    cfg = O.Config(1, 30, 32, 10, 30, 30, np.array([0.5], np.float32))
    with pytest.raises(O.OracleError) as e:
        O.encode(cfg, x)
    assert e.value.code == O.ERR_NONFINITE
    x[0, 1, 17, 5] = np.nan
    with pytest.raises(O.OracleError) as e:
        O.encode(cfg, x)
    assert e.value.code == O.ERR_NONFINITE
    for bad in [O.Config(1, 30, 48, 10, 30, 30, np.array([0.5], np.float32)),
                O.Config(1, 30, 32, 0, 30, 30, np.array([0.5], np.float32)),
                O.Config(1, 30, 32, 10, 30, 30, np.array([2.0 ** -10], np.float32)),
                O.Config(1, 30, 32, 10, 30, 30, np.array([np.nan], np.float32))]:
        with pytest.raises(O.OracleError) as e:
            O.geometry(bad)
        assert e.value.code == O.ERR_INVALID_ARG


# --------------------------------------------------------------------------
# histogram and coded size
# --------------------------------------------------------------------------

def test_histograms_match_bincount():
    w = synth.small("t", 2, 97, 64, seed=6)
    x = w.generate().numpy()
    cfg = O.Config(2, 97, 64, 10, 50, 50, O.layer_steps(2))
    sc = O.anchor_scales(cfg, x)
    _, q = O.quantize(cfg, x, sc)
    h = O.histograms(cfg, q)
    am = O.anchor_mask(cfg)
    sym = np.where(np.abs(q) <= 127, q + 127, 255)[:, :, ~am, :]
    for l in range(2):
        for kv in range(2):
            for c in range(64):
                ref = np.bincount(sym[l, kv, :, c], minlength=256)
                assert np.array_equal(h[(l * 2 + kv) * 64 + c], ref)


def test_coded_size_within_one_percent_of_empirical_entropy():
    w = synth.small("t", 2, 2048, 256, seed=0)
    x = w.generate().numpy()
    cfg = O.Config(2, 2048, 256, 10, 2048, 1536, O.layer_steps(2))
    enc = O.encode(cfg, x, nthreads=4)
    sc = O.anchor_scales(cfg, x)
    _, q = O.quantize(cfg, x, sc)
    h = O.histograms(cfg, q).astype(np.float64)
    N = h.sum(1, keepdims=True)
    H = -(h * np.log2(np.where(h > 0, h / np.maximum(N, 1), 1))).sum()
    geo = O.geometry(cfg)
    streams = geo["n_streams"]
    body = 8 * enc.payload.size - 32 * 32 * streams - 16 * 8 * streams  # minus flush and padding slack
    assert body <= 1.01 * H
    assert 8 * enc.payload.size >= H - 16 * 32 * streams


# --------------------------------------------------------------------------
# generator sanity (the synthetic data has the token locality the pages describe)
# --------------------------------------------------------------------------

def test_generator_delta_variance_ratio():
    x = synth.ar1_kv(2, 4000, 256, 0.95, 2, seed=0).numpy().astype(np.float64)
    G = 10
    anc = x[:, :, ::G, :]
    d = (x.reshape(2, 2, 400, G, 256) - anc[:, :, :, None, :])[:, :, :, 1:, :]
    ratio = x.var(axis=2).mean() / d.reshape(2, 2, -1, 256).var(axis=2).mean()
    rho = 0.95
    expect = 1.0 / (2 * (1 - np.mean([rho ** k for k in range(1, G)])))
    assert abs(ratio - expect) / expect < 0.1
    # outliers: n_outlier channels per layer carry ~20x scale
    std = x.std(axis=2).mean(axis=1)  # [L][C]
    for l in range(2):
        assert (std[l] > 8 * np.median(std[l])).sum() == 2


def test_threaded_encode_decode_equal_single_threaded():
    w = synth.small("t", 3, 700, 64, seed=8)
    x = w.generate().numpy()
    cfg = O.Config(3, 700, 64, 10, 300, 128, O.layer_steps(3))
    e1 = O.encode(cfg, x, nthreads=1)
    e4 = O.encode(cfg, x, nthreads=4)
    for f in ["anchors", "scales", "tables", "table_off", "payload", "stream_off", "escapes", "esc_off"]:
        assert np.array_equal(getattr(e1, f), getattr(e4, f)), f
    assert np.array_equal(O.decode(cfg, e1, 1), O.decode(cfg, e4, 3))
