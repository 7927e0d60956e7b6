"""Host logic: the create-time work splits of the absorbing kernels
(mla_split.cpp), for every head count 1..128 and several CTA counts.

A decode step (page "mla.query", class MlaQuery) streams each weight byte
once, so it lasts as long as its most loaded CTA.  Each split must hand out
every head, task and rope row exactly once, in contiguous runs, never give a
cluster pair more than two heads, and keep every CTA within one rope unit of
the larger of the even share and its own head or task bytes.  The splits are
compiled from the library's source with a small driver (tests/split_driver.cpp);
no GPU is needed."""

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "mla_query_projection_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

TASK = 16 * 1536 * 2 + 16 * 512 * 2  # one task: 16 Q_B rows and their 16 W_UK rows
ROW = 1536 * 2                       # one rope row of W_QB
HEAD_BOXES, ROPE_BOXES, SINGLE_BOXES = 16, 12, 6  # wide kernel, 16 KiB boxes per CTA


@pytest.fixture(scope="module")
def splits(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")):
        pytest.skip("needs g++ and the CUDA headers")
    exe = str(tmp_path_factory.mktemp("splits") / "split_driver")
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                    "-I", CUDA_INC, os.path.join(HERE, "split_driver.cpp"),
                    os.path.join(CSRC, "mla_split.cpp"), "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    rows = {"abs": [], "pair": [], "pairf": [], "pairmax": [], "fmafirst": [], "wide": [],
            "small": [], "choose": []}
    for line in out.splitlines():
        f = line.split()
        rows[f[0]].append((int(f[1]), int(f[2]), [int(x) for x in f[3:]]))
    assert all(len(rows[k]) == 9 * 128 for k in ("abs", "pair", "pairf", "wide", "choose"))
    assert len(rows["small"]) == 3 * 9 * 128
    return rows


def runs(bounds, total):
    """Contiguous runs [bounds[i], bounds[i+1]) covering [0, total) once."""
    assert bounds[0] == 0 and bounds[-1] == total, (bounds[0], bounds[-1], total)
    assert all(b <= c for b, c in zip(bounds, bounds[1:]))
    return [c - b for b, c in zip(bounds, bounds[1:])]


def test_absorbing_split(splits):
    for heads, ctas, v in splits["abs"]:
        tasks = runs(v[:ctas + 1], 8 * heads)
        rope = runs(v[ctas + 1:], 64 * heads)
        assert max(tasks) - min(tasks) <= 1, (heads, ctas)  # tasks evenly
        mean = (8 * heads * TASK + 64 * heads * ROW) / ctas
        for t, r in zip(tasks, rope):
            assert t * TASK + r * ROW < max(mean, t * TASK) + ROW, (heads, ctas)


@pytest.mark.parametrize("order", ["pair", "pairf"])
def test_paired_split(splits, order):
    for heads, ctas, v in splits[order]:
        pairs = ctas // 2
        ok, head, rope = v[0], v[1:pairs + 2], v[pairs + 2:]
        # refused exactly when some pair would need a third head
        assert ok == (heads <= 2 * pairs), (heads, ctas)
        if not ok:
            continue
        nh = runs(head, heads)
        assert max(nh) <= 2
        if order == "pair" or heads > pairs:  # evenly: counts differ by one at most
            assert max(nh) - min(nh) <= 1, (heads, ctas)
        else:  # heads first: one head on each of the first `heads` pairs
            assert nh == [1] * heads + [0] * (pairs - heads), (heads, ctas)
        rows = runs(rope, 64 * heads)
        mean = (heads * 8 * TASK + 64 * heads * ROW) / ctas
        for i, r in enumerate(rows):
            own = nh[i // 2] * 4 * TASK  # each CTA takes 4 of a head's 8 tasks
            assert own + r * ROW < max(mean, own) + ROW, (heads, ctas, i)


def wide_fields(heads, ctas, v):
    """(ok, ndouble, heads per pair, two-head units per pair, one-head units
    per pair) of a wide split line."""
    pairs = ctas // 2
    ok, nd = v[0], v[1]
    head, dbl, sgl = v[2:pairs + 3], v[pairs + 3:2 * pairs + 4], v[2 * pairs + 4:]
    if not ok:
        return ok, nd, None, None, None
    singles = max(0, heads - 2 * nd)
    return ok, nd, runs(head, heads), runs(dbl, nd), runs(sgl, singles)


def wide_cost(nh, d, s):
    """The planner's estimate in quarter boxes: 4 a 128-row box (16 per head,
    12 per two-head unit), 5 a 64-row box (6 per one-head unit)."""
    return 4 * HEAD_BOXES * nh + 4 * ROPE_BOXES * d + 5 * SINGLE_BOXES * s


def test_paired_split_max_bytes(splits):
    """pair_split_max_bytes is the most loaded CTA of the heads-first split:
    half a head's four tasks per head of its pair plus its rope rows."""
    most = {(h, c): v[0] for h, c, v in splits["pairmax"]}
    n = 0
    for heads, ctas, v in splits["pairf"]:
        if not v[0]:
            continue
        pairs = ctas // 2
        nh = runs(v[1:pairs + 2], heads)
        rows = runs(v[pairs + 2:], 64 * heads)
        loads = [nh[i // 2] * 4 * TASK + r * ROW for i, r in enumerate(rows)]
        assert most[(heads, ctas)] == max(loads), (heads, ctas)
        n += 1
    assert n > 600


def test_one_token_dispatch_boundary(splits):
    """One token takes the FMA kernel where its most loaded CTA carries at
    most 80 % of the paired kernel's: on 152 SMs with GB300's cluster limits
    that is every head count up to 36 (clusters of 8 or 4 split a head four
    or eight ways; 37 heads no longer fit 36 clusters of four), and none
    above (both kernels then put whole half-heads on their most loaded CTA)."""
    got = {h: v for h, c, v in splits["fmafirst"]}
    assert sorted(got) == list(range(1, 129))
    for h, (fm, pm, fma) in got.items():
        assert fma == (5 * fm <= 4 * pm), h
        assert fma == (h <= 36), (h, fm, pm)


def test_wide_split(splits):
    """Every head's rope rows are covered once: two-head units cover heads
    0 .. 2 ndouble - 1, one-head units the rest; no pair has more than two
    heads; and no pair's estimated time exceeds the least loaded pair's by
    more than the largest unit (each unit went to the least loaded pair)."""
    for heads, ctas, v in splits["wide"]:
        pairs = ctas // 2
        ok, nd, nh, d, s = wide_fields(heads, ctas, v)
        assert ok == (heads <= 2 * pairs), (heads, ctas)
        if not ok:
            continue
        assert 0 <= nd <= (heads + 1) // 2
        assert max(nh) <= 2
        assert sum(d) == nd and sum(s) == max(0, heads - 2 * nd)
        cost = [wide_cost(*x) for x in zip(nh, d, s)]
        # a pair that got a unit was the least loaded when it did
        for c in range(pairs):
            if d[c] + s[c]:
                assert cost[c] <= min(cost) + 4 * ROPE_BOXES, (heads, ctas, c)


def test_wide_split_shapes_on_76_pairs(splits):
    """The cases the wide kernel's measurements rest on (152 CTAs): mixing the
    rope-unit shapes brings 127 and 128 heads from 44 boxes on the most
    loaded CTA (two-head units only) to 40; 64 heads stay at 22 (one-head
    units only gave 22, two-head units 28); 16 heads at 16."""
    got = {h: v for h, c, v in splits["wide"] if c == 152}
    for heads, most in ((64, 22), (127, 40), (128, 40), (16, 16)):
        ok, nd, nh, d, s = wide_fields(heads, 152, got[heads])
        assert ok
        boxes = [HEAD_BOXES * n + ROPE_BOXES * a + SINGLE_BOXES * b for n, a, b in zip(nh, d, s)]
        assert max(boxes) == most, (heads, max(boxes))


SMALL_ROWS = 1536 * 2 + 512 * 2  # one nope row of the small-batch kernel: Q_B row + W_UK row


def test_small_split(splits):
    """Clusters of K CTAs (2, 4, 8) own whole heads, at most two each; rank r
    of a cluster takes 128/K nope rows of each; rope rows fill every CTA to
    an even share, so no CTA is more than one rope row above the larger of
    the share and its own nope bytes.  The reported maximum is exact."""
    seen = 0
    for heads, ctas, v in splits["small"]:
        k, ok, most = v[0], v[1], v[2]
        if ctas < k:
            assert not ok
            continue
        groups = ctas // k
        assert ok == (heads <= 2 * groups), (heads, ctas, k)
        if not ok:
            continue
        seen += 1
        head, rope = v[3:groups + 4], v[groups + 4:]
        nh = runs(head, heads)
        assert max(nh) <= 2
        rows = runs(rope, 64 * heads)
        mean = (heads * 128 * SMALL_ROWS + 64 * heads * ROW) / ctas
        loads = []
        for i, r in enumerate(rows):
            own = nh[i // k] * (128 // k) * SMALL_ROWS
            loads.append(own + r * ROW)
            assert own + r * ROW < max(mean, own) + ROW, (heads, ctas, k, i)
        assert max(loads) == most, (heads, ctas, k)
    assert seen > 1000


def test_small_split_choice(splits):
    """The cluster size chosen is the one with the fewest bytes on the most
    loaded CTA (ties: the smaller cluster); on 152 SMs: 64 and 128 heads take
    pairs, 16 heads clusters of 8 (64 KiB of nope rows a CTA instead of 256)."""
    small = {(h, c, v[0]): v for h, c, v in splits["small"]}
    for heads, sms, v in splits["choose"]:
        ctas, k, most = v
        cands = []
        for kk in (2, 4, 8):
            row = small.get((heads, (sms // kk) * kk, kk))
            if row is not None and row[1]:
                cands.append((row[2], kk))
        if not cands:
            assert ctas == 0, (heads, sms)
            continue
        best = min(m for m, _ in cands)
        assert most == best, (heads, sms)
        assert k == min(kk for m, kk in cands if m == best), (heads, sms)
    got = {h: v for h, s_, v in splits["choose"] if s_ == 152}
    assert got[64][1] == 2 and got[128][1] == 2 and got[16][1] == 8
    assert got[16][2] < 80 * 1024
