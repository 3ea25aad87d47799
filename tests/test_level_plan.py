"""Bandwidth-adaptive level choice per chunk (cg_plan_levels, host only).

The planner follows the chunked multi-level streaming of the CacheGen pages
("CacheGen vs 传统量化KV缓存压缩技术深度对比与性能测试", §2.2): every chunk is
stored at several quality levels and the sender picks, chunk by chunk, the
best quality whose transfer plus decode still meets the deadline.  Checked
here against a hand-worked case, limiting cases, invariants (feasibility,
monotonicity in the deadline) and a plain Python simulation of the same rule.
"""
import math

import numpy as np
import pytest

from kv_cache_compression_decode_gb300 import codec as C


def _py_plan(nbytes, dec, bw, slot_s, slo):
    """The rule of include/cg.h written out step by step."""
    n, Q = nbytes.shape
    low = Q - 1

    def transfer_end(t0, b):
        t, rem = t0, float(b)
        k = min(int(math.floor(t / slot_s)), len(bw) - 1)
        while k + 1 < len(bw):
            end = (k + 1) * slot_s
            if end > t:
                cap = (end - t) * bw[k]
                if cap >= rem:
                    return t + rem / bw[k]
                rem -= cap
                t = end
            k += 1
        return t + rem / bw[-1]

    def predict(i, q, t_link, t_gpu, b):
        tl = t_link + nbytes[i, q] / b
        tg = max(tl, t_gpu) + dec[i, q]
        for j in range(i + 1, n):
            tl += nbytes[j, low] / b
            tg = max(tl, tg) + dec[j, low]
        return tg

    t_link = t_gpu = 0.0
    b = bw[0]
    levels, arrive, done = [], [], []
    for i in range(n):
        q = next((c for c in range(Q - 1) if predict(i, c, t_link, t_gpu, b) <= slo), low)
        a = transfer_end(t_link, nbytes[i, q])
        if a > t_link:
            b = nbytes[i, q] / (a - t_link)
        t_gpu = max(a, t_gpu) + dec[i, q]
        t_link = a
        levels.append(q)
        arrive.append(a)
        done.append(t_gpu)
    return np.array(levels), np.array(arrive), np.array(done), t_gpu


def test_hand_worked_three_chunks():
    # 10 B/s, sizes 100/50/25 per level, no decode time, deadline 17.5 s:
    # chunk 0 at level 0 ends at 10 s and leaves 2 x 2.5 s for the rest at the
    # lowest level (15 s); chunk 1 at level 0 would end at 20 s, at level 1
    # at 15 s (+2.5 s = 17.5 s); chunk 2 fits only at level 2.
    nb = np.array([[100, 50, 25]] * 3)
    p = C.cg_plan_levels(nb, np.zeros((3, 3)), np.array([10.0]), 1.0, 17.5)
    assert p.levels.tolist() == [0, 1, 2]
    assert np.allclose(p.arrive_s, [10.0, 15.0, 17.5]) and p.finish_s == pytest.approx(17.5)


def test_limits_of_bandwidth():
    rng = np.random.default_rng(1)
    nb = np.sort(rng.integers(1000, 10**6, (8, 3)), axis=1)[:, ::-1].copy()
    dec = np.full((8, 3), 1e-3)
    assert C.cg_plan_levels(nb, dec, np.array([1e15]), 1.0, 1.0).levels.tolist() == [0] * 8
    assert C.cg_plan_levels(nb, dec, np.array([1.0]), 1.0, 1.0).levels.tolist() == [2] * 8


def test_decode_time_is_pipelined_with_transfer():
    # transfer 1 s per chunk, decode 2 s per chunk: the GPU is the bottleneck
    p = C.cg_plan_levels(np.array([[10]] * 3), np.array([[2.0]] * 3), np.array([10.0]), 1.0, 100.0)
    assert np.allclose(p.arrive_s, [1, 2, 3]) and np.allclose(p.done_s, [3, 5, 7]) and p.finish_s == 7.0


@pytest.mark.parametrize("seed", range(12))
def test_matches_python_rule_on_traces(seed):
    rng = np.random.default_rng(seed)
    n, Q = int(rng.integers(1, 13)), int(rng.integers(1, 5))
    nb = np.sort(rng.integers(1, 10**7, (n, Q)), axis=1)[:, ::-1].astype(np.float64)
    dec = rng.uniform(0, 0.02, (n, Q))
    bw = rng.uniform(1e7, 3e8, int(rng.integers(1, 9)))
    slot_s = float(rng.uniform(0.005, 0.1))
    slo = float(rng.uniform(0.05, 2.0))
    got = C.cg_plan_levels(nb.astype(np.uint64), dec, bw, slot_s, slo)
    lv, ar, dn, fin = _py_plan(nb, dec, bw, slot_s, slo)
    assert got.levels.tolist() == lv.tolist()
    assert np.allclose(got.arrive_s, ar, rtol=1e-12) and np.allclose(got.done_s, dn, rtol=1e-12)
    assert got.finish_s == pytest.approx(fin, rel=1e-12)


def test_constant_bandwidth_meets_a_feasible_deadline_and_is_monotone():
    rng = np.random.default_rng(7)
    nb = np.sort(rng.integers(10**5, 10**7, (10, 3)), axis=1)[:, ::-1].copy()
    dec = rng.uniform(0, 0.01, (10, 3))
    bw = np.array([5e8])
    low = C.cg_plan_levels(nb, dec, bw, 1.0, 0.0)  # nothing fits: all lowest
    assert low.levels.tolist() == [2] * 10
    prev = -1
    for slo in np.linspace(low.finish_s, 3 * low.finish_s, 25):
        p = C.cg_plan_levels(nb, dec, bw, 1.0, float(slo))
        assert p.finish_s <= slo * (1 + 1e-12)
        sent = int(sum(nb[i, q] for i, q in enumerate(p.levels)))
        assert sent >= prev
        prev = sent


def test_bandwidth_drop_lowers_later_levels():
    nb = np.array([[4e6, 2e6, 1e6]] * 6, dtype=np.uint64)
    dec = np.zeros((6, 3))
    steady = C.cg_plan_levels(nb, dec, np.array([1e8]), 0.01, 0.2)
    drop = C.cg_plan_levels(nb, dec, np.array([1e8, 1e8, 1e8, 1e8, 1e7]), 0.01, 0.2)
    # 0.2 s at 100 MB/s carries 20 MB: four chunks at level 0, two at level 1
    assert steady.levels.tolist() == [0, 0, 0, 0, 1, 1] and steady.finish_s == pytest.approx(0.2)
    # the link falls to 10 MB/s from 40 ms on: chunk 1 (planned at 100 MB/s)
    # is caught by the drop, and every later chunk goes to the lowest level
    assert drop.levels.tolist() == [0, 0, 2, 2, 2, 2]
    assert (drop.levels >= steady.levels).all()


@pytest.mark.parametrize("bad", ["bw0", "bwnan", "slot0", "none", "decneg"])
def test_invalid_arguments(bad):
    nb, dec, bw, slot = np.array([[10, 5]]), np.zeros((1, 2)), np.array([1.0]), 1.0
    if bad == "bw0":
        bw = np.array([0.0])
    elif bad == "bwnan":
        bw = np.array([np.nan])
    elif bad == "slot0":
        slot = 0.0
    elif bad == "none":
        nb, dec = np.zeros((0, 2)), np.zeros((0, 2))
    elif bad == "decneg":
        dec = np.array([[0.0, -1.0]])
    with pytest.raises(C.CodecError):
        C.cg_plan_levels(nb, dec, bw, slot, 1.0)
