"""The benchmark steps' two-stream schedules, checked on the host: every pair of
ops that touch the same buffer (one of them writing it) is ordered by the
schedule's happens-before relation -- program order on each stream, the
cross-stream waits of the step's WAITS, the fork at the step's start and the
join at its end -- and the ops sharing a context run on one stream.

The buffers each op reads and writes are listed here from the steps' data flow
(quantize X and W, fprop, quantize dY, dgrad, wgrad, and for the NVFP4 step the
DGE on W).  A context's NVFP4 amax scratch is checked separately: the side ops
pass the step's side context, so each context's calls stay on one stream.  Both
steps are checked: the 7B FFN step the benchmark's headline times (bench.FfnStep)
and the LLaMA-1B NVFP4 step (bench.Step).
"""
import itertools
from types import SimpleNamespace

import pytest

import bench

READS = {
    "quant_x_dual": {"X"},
    "quant_w_dual": {"W"},
    "fprop": {"xq", "wq"},
    "quant_dy_dual": {"dY"},
    "dgrad": {"dyq_n", "wq_t"},
    "wgrad": {"dyq_m", "xq_t"},
    "dge": {"W", "wq", "dW"},
}
WRITES = {
    "quant_x_dual": {"xq", "xq_t"},
    "quant_w_dual": {"wq", "wq_t"},
    "fprop": {"Y"},
    "quant_dy_dual": {"dyq_n", "dyq_m"},
    "dgrad": {"dX"},
    "wgrad": {"dW"},
    "dge": {"dWd"},
}


STEPS = {"llama": bench.Step, "ffn": bench.FfnStep}
FFN_OPS = ("quant_x_dual", "quant_w_dual", "fprop", "quant_dy_dual", "dgrad", "wgrad")


def _op_names(cls=bench.Step):
    step = object.__new__(cls)             # the op list only; no buffers are touched
    step.fp4 = None
    step.p_dy_n = step.p_w_t = step.p_dy_m = step.p_x_t = SimpleNamespace()
    step.p_rows = step.p_cols = SimpleNamespace()
    return [name for name, _ in step.ops(0)]


def _schedule(names, cls=bench.Step):
    """(stream of each op, happens-before as a set of (earlier, later) pairs)."""
    stream = {n: ("side" if n in cls.SIDE else "main") for n in names}
    hb = set()
    for a, b in itertools.combinations(names, 2):          # enqueue order on one stream
        if stream[a] == stream[b]:
            hb.add((a, b))
    for later, earlier in cls.WAITS.items():               # a side wait: `later` after `earlier`
        hb.add((earlier, later))
    # transitive closure
    changed = True
    while changed:
        changed = False
        for (a, b), (c, d) in itertools.product(list(hb), list(hb)):
            if b == c and (a, d) not in hb:
                hb.add((a, d))
                changed = True
    return stream, hb


def _unordered_conflicts(names, hb):
    out = []
    for a, b in itertools.combinations(names, 2):
        conflict = (WRITES[a] & (READS[b] | WRITES[b])) | (WRITES[b] & READS[a])
        if conflict and (a, b) not in hb and (b, a) not in hb:
            out.append((a, b, sorted(conflict)))
    return out


@pytest.mark.parametrize("which", sorted(STEPS))
def test_every_conflicting_pair_is_ordered(which):
    cls = STEPS[which]
    names = _op_names(cls)
    assert set(names) == (set(READS) if which == "llama" else set(FFN_OPS))
    _, hb = _schedule(names, cls)
    assert _unordered_conflicts(names, hb) == []


@pytest.mark.parametrize("which", sorted(STEPS))
def test_readers_come_after_their_producers(which):
    cls = STEPS[which]
    names = _op_names(cls)
    _, hb = _schedule(names, cls)
    producer = {buf: op for op, bufs in WRITES.items() for buf in bufs}
    for op in names:
        for buf in READS[op]:
            if buf in producer:
                assert (producer[buf], op) in hb, f"{op} may read {buf} before {producer[buf]} writes it"


@pytest.mark.parametrize("which", sorted(STEPS))
def test_each_context_serves_one_stream(which):
    cls = STEPS[which]
    names = _op_names(cls)
    stream, _ = _schedule(names, cls)
    # side ops pass the side context, the others the default one
    assert {stream[n] for n in names if n in cls.SIDE} == {"side"}
    assert {stream[n] for n in names if n not in cls.SIDE} == {"main"}


@pytest.mark.parametrize("which", sorted(STEPS))
def test_the_schedule_overlaps_independent_work(which):
    """The point of the second stream: the two forward quantizations, and dgrad
    with wgrad, are not ordered against each other."""
    cls = STEPS[which]
    names = _op_names(cls)
    _, hb = _schedule(names, cls)
    pairs = [("quant_x_dual", "quant_w_dual"), ("dgrad", "wgrad")] + ([("dgrad", "dge")] if which == "llama" else [])
    for a, b in pairs:
        assert (a, b) not in hb and (b, a) not in hb


def test_a_missing_wait_is_caught(monkeypatch):
    """Planting a schedule mistake (wgrad no longer waits for dY's quantization)
    makes the race check fail."""
    monkeypatch.setattr(bench.Step, "WAITS", {"fprop": "quant_w_dual"})
    names = _op_names()
    _, hb = _schedule(names)
    assert ("quant_dy_dual", "wgrad", ["dyq_m"]) in _unordered_conflicts(names, hb)
