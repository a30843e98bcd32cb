"""Host checks of the work queues the fused kernel runs (build_queues, the
builder shared by the host-split path and the device plan kernel), compiled
for the host from the kernel header and run on random expert splits:

- every item of every non-empty expert is in exactly one segment (amax and
  encode items for the two-pass NVFP4 recipe, single-pass items otherwise);
- queue 1 lists the experts in the required order (by decreasing size,
  stable, for two passes; by index otherwise);
- static interleave: an expert's encode segments come after all of its amax
  items and after `lookahead` further amax items (or at the tail), the order
  the deadlock-freedom argument rests on;
- ready-first: queue 2 holds one encode segment per expert, in queue 1's order.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
K_SINGLE, K_P1, K_P2 = 0, 1, 2


@pytest.fixture(scope="module")
def harness():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    d = tempfile.mkdtemp()
    exe = os.path.join(d, "plan_harness")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I" + os.path.join(ROOT, "include"),
                    "-I" + os.path.join(ROOT, "nvfp4_quantization_grouped_gb300", "csrc"),
                    "-o", exe, os.path.join(ROOT, "tests", "native", "plan_harness.cu")], check=True)
    yield exe
    shutil.rmtree(d, ignore_errors=True)


def run_cases(exe, cases, parallel=False):
    text = "".join(f"{len(m)} {ns} {ns2} {int(tp)} {int(rf)} {la} " + " ".join(map(str, m)) + "\n"
                   for m, ns, ns2, tp, rf, la in cases)
    args = [exe, "parallel"] if parallel else [exe]
    out = subprocess.run(args, input=text, capture_output=True, text=True, check=True).stdout.split("\n")
    res, i = [], 0
    for _ in cases:
        n1, s1, n2, sn = map(int, out[i].split())
        segs = [tuple(map(int, out[i + 1 + k].split())) for k in range(sn)]
        res.append((n1, s1, n2, sn, segs))
        i += 1 + sn
    return res


def check(m, n_slabs, n_slabs2, two_pass, ready_first, lookahead, result):
    n1, s1, n2, sn, segs = result
    items = [((int(x) + 127) // 128) * n_slabs for x in m]
    items2 = [((int(x) + 127) // 128) * n_slabs2 for x in m]    # encode items
    nonempty = [e for e in range(len(m)) if m[e] > 0]
    order = sorted(nonempty, key=lambda e: -m[e]) if two_pass else nonempty   # sorted() is stable
    q1, q2 = segs[:s1], segs[s1:]
    # contiguous queues; a segment's length is the next start (or the queue size) minus its start
    def spans(q, total):
        starts = [s[0] for s in q]
        assert starts == sorted(starts) and (not q or starts[0] == 0)
        return [(q[k][1], q[k][2], q[k][3], (starts[k + 1] if k + 1 < len(q) else total) - starts[k], starts[k])
                for k in range(len(q))]
    sp1, sp2 = spans(q1, n1), spans(q2, n2)
    assert all(c > 0 for *_, c, _ in sp1 + sp2)
    cover = {}
    for kind, e, first, cnt, _ in sp1 + sp2:
        cover.setdefault((kind, e), []).append((first, cnt))
    kinds = (K_P1, K_P2) if two_pass else (K_SINGLE,)
    for e in nonempty:
        for kind in kinds:
            got = sorted(cover.pop((kind, e)))
            pos = 0
            for first, cnt in got:
                assert first == pos, (e, kind, got)
                pos += cnt
            want = items2[e] if kind == K_P2 else items[e]
            assert pos == want, (e, kind, pos, want)
    assert not cover, cover
    first_kind = K_P1 if two_pass else K_SINGLE
    seen = []
    for kind, e, *_ in sp1:
        if kind == first_kind and e not in seen:
            seen.append(e)
    assert seen == order
    if two_pass and ready_first:
        assert [e for kind, e, *_ in sp2] == order and all(kind == K_P2 for kind, *_ in sp2)
        assert n2 == sum(items2[e] for e in order)
    elif two_pass:
        assert not sp2
        p1_before = 0
        p1_end = {}
        total_p1 = sum(items[e] for e in order)
        for kind, e, first, cnt, _ in sp1:
            if kind == K_P1:
                p1_before += cnt
                if first + cnt == items[e]:
                    p1_end[e] = p1_before
            else:
                assert e in p1_end, "encode items before the expert's amax items"
                assert p1_before >= min(p1_end[e] + lookahead, total_p1)


def _random_cases():
    rng = np.random.default_rng(12)
    cases = []
    for _ in range(300):
        E = int(rng.integers(1, 257))
        kind = rng.integers(0, 4)
        if kind == 0:
            m = rng.integers(0, 5000, E)
        elif kind == 1:
            m = rng.multinomial(int(rng.integers(0, 200000)), rng.dirichlet(np.full(E, 0.3)))
        elif kind == 2:
            m = np.where(rng.random(E) < 0.5, 0, rng.integers(1, 300, E))
        else:
            m = np.full(E, int(rng.integers(0, 1000)))
        n_slabs = int(rng.choice([1, 2, 4, 8, 16]))
        n_slabs2 = n_slabs * int(rng.choice([1, 1, 2, 4]))       # encode items: the same or smaller
        two_pass = bool(rng.integers(0, 2))
        ready_first = bool(rng.integers(0, 2))
        lookahead = int(rng.choice([0, 1, 7, 152, 304, 1000]))
        cases.append(([int(x) for x in m], n_slabs, n_slabs2, two_pass, ready_first, lookahead))
    return cases


def test_queues_cover_order_and_lookahead(harness):
    cases = _random_cases()
    for case, res in zip(cases, run_cases(harness, cases)):
        check(*case, res)


def test_parallel_build_equals_serial(harness):
    """The plan kernel's parallel queue build (one position of the order per
    thread, prefix sums between its steps) gives the serial builder's tables
    segment for segment: every case of the cover test, plus edge cases (no
    non-empty expert, one expert, 256 experts, lookahead 0 and larger than
    every queue, encode items the size of the amax items or smaller)."""
    cases = _random_cases()
    for tp, rf in ((False, False), (True, False), (True, True)):
        for la in (0, 1, 5, 304, 10 ** 6):
            cases.append(([0, 0, 0], 2, 4, tp, rf, la))
            cases.append(([1000], 4, 8, tp, rf, la))
            cases.append(([128] * 256, 1, 1, tp, rf, la))
            cases.append(([1, 0, 129, 256, 0, 7], 8, 8, tp, rf, la))
    serial = run_cases(harness, cases)
    par = run_cases(harness, cases, parallel=True)
    for case, a, b in zip(cases, serial, par):
        assert a == b, case[1:]
