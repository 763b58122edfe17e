"""C ABI exports and the planner/validator, on the CPU (no GPU calls)."""
import ctypes
import os
import re

import pytest

import synthetic as S
import tile_scheduled_persistent_gb300 as tsp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    tsp.build()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(tiles_[a-z_0-9]+)\s*\(", src))
    return names


def test_library_exports_every_declared_function():
    declared = _declared()
    assert declared >= set(tsp.EXPORTS)
    lib = ctypes.CDLL(tsp._LIB_PATH)
    for name in sorted(declared):
        assert hasattr(lib, name), name


def test_status_strings():
    lib = tsp.lib()
    for code in range(-8, 1):
        assert lib.tiles_status_string(code)
    assert lib.tiles_status_string(-99) == b"unknown status"


def _sched(name="llama1b", n=152, **opts):
    return tsp.Schedule(tsp.ModelDesc.from_config(S.CONFIGS[name]), n, tsp.make_opts(**opts))


@pytest.mark.parametrize("name", list(S.CONFIGS))
@pytest.mark.parametrize("scheduler", [0, 1, 2])
def test_schedules_validate_and_balance(name, scheduler):
    cfg = S.CONFIGS[name]
    s = _sched(name, scheduler=scheduler)
    st, why = s.validate()
    assert st == 0, why
    b = s.cta_bytes(cfg.start_pos)
    assert abs(sum(b) - cfg.algorithmic_bytes_per_token()) / cfg.algorithmic_bytes_per_token() < 0.01
    if name != "tiny":
        assert max(b) / (sum(b) / len(b)) < 1.03          # byte balance across CTAs


def test_weight_rows_balanced_to_one_row_per_phase():
    s = _sched("llama1b")
    tasks, off = s.tasks()
    counts = {}
    for c in range(len(off) - 1):
        for i in range(off[c], off[c + 1]):
            t = tasks[i]
            if t.op in (1, 4, 5, 6, 7):
                counts.setdefault((t.op, t.layer), []).append(t.end - t.begin)
    for k, v in counts.items():
        assert max(v) - min(v) <= 1, k


def _mutate_and_expect(mutator, expect):
    s = _sched("tiny", n=16, scheduler=1)   # the counters schedule: every tile waits
    tasks, off = s.tasks()
    mutator(tasks, off)
    st, why = s.validate()
    assert st == -3, f"mutation accepted ({why})"
    assert expect in why, why


def test_rejects_dropped_rows():
    def m(tasks, off):
        t = tasks[off[3]]
        t.end = t.end - 1 if t.end - t.begin > 1 else t.end
        t.begin += 0 if t.end - t.begin > 0 else 0
    _mutate_and_expect(m, "not covered")


def test_rejects_duplicated_rows():
    def m(tasks, off):
        tasks[off[3]].begin = max(0, tasks[off[3]].begin - 1)
    _mutate_and_expect(m, "covered twice")


def test_rejects_wrong_wait_target():
    def m(tasks, off):
        tasks[off[2] + 1].wait_add += 1
    _mutate_and_expect(m, "wait target")


def test_rejects_wait_on_a_later_phase():
    def m(tasks, off):
        t = tasks[off[2] + 1]
        t.wait_ctr = (t.signal_ctr + 1) % 13     # a counter signalled after this phase
    _mutate_and_expect(m, "wait")


def test_flags_schedule_waits_only_where_inputs_are_untagged():
    s = _sched("llama1b", scheduler=2)
    tasks, off = s.tasks()
    NO = 0xFFFF
    for c in range(len(off) - 1):
        for i in range(off[c], off[c + 1]):
            t = tasks[i]
            waits = t.op == 1 and t.layer == 0                      # first Q/K/V of a step
            assert (t.wait_ctr != NO) == waits, (t.op, t.layer)
            assert (t.signal_ctr != NO) == (t.op == 7)               # the LM head signals


def _mutate_flags_and_expect(mutator, expect):
    s = _sched("tiny", n=16, scheduler=2)
    tasks, off = s.tasks()
    mutator(tasks, off)
    st, why = s.validate()
    assert st == -3, f"mutation accepted ({why})"
    assert expect in why, why


def test_flags_rejects_a_first_qkv_tile_that_does_not_wait():
    def m(tasks, off):
        for i in range(len(tasks)):
            if tasks[i].op == 1 and tasks[i].layer == 0:
                tasks[i].wait_ctr = 0xFFFF
                return
    _mutate_flags_and_expect(m, "without a wait")


def test_flags_rejects_an_attention_cta_that_does_not_signal_the_lm_head():
    # the LM-head release of the same CTA is what orders its K/V writes
    def m(tasks, off):
        c = next(c for c in range(len(off) - 1)
                 if any(tasks[i].op == 2 for i in range(off[c], off[c + 1])))
        for i in range(off[c], off[c + 1]):
            if tasks[i].op == 7:
                tasks[i].signal_ctr = 0xFFFF
    _mutate_flags_and_expect(m, "")


def test_rejects_out_of_range_layer_and_op():
    def m(tasks, off):
        tasks[off[1]].layer = 99
    _mutate_and_expect(m, "layer")

    def m2(tasks, off):
        tasks[off[1]].op = 42
    _mutate_and_expect(m2, "unknown op")


def test_rejects_out_of_order_tasks():
    def m(tasks, off):
        a, b = tasks[off[5]], tasks[off[5] + 2]
        for f, _ in tsp.Task._fields_:
            x, y = getattr(a, f), getattr(b, f)
            setattr(a, f, y)
            setattr(b, f, x)
    _mutate_and_expect(m, "order")


def test_rejects_unsupported_shapes():
    cfg = S.CONFIGS["tiny"]
    for bad in (dict(head_dim=96), dict(n_kv_heads=3), dict(hidden=260)):
        from dataclasses import replace
        d = tsp.ModelDesc.from_config(replace(cfg, **bad))
        with pytest.raises(tsp.TilesError) as e:
            tsp.Schedule(d, 16)
        assert e.value.status in (-1, -2)


def test_rejects_bad_options():
    d = tsp.ModelDesc.from_config(S.CONFIGS["tiny"])
    for o in (tsp.make_opts(scheduler=7), tsp.make_opts(slot_bytes=1000),
              tsp.make_opts(ring_slots=1)):
        with pytest.raises(tsp.TilesError):
            tsp.Schedule(d, 16, o)
    with pytest.raises(tsp.TilesError):                      # unknown flag bits
        tsp.Schedule(d, 16, tsp.make_opts(flags=2))
    st, why = tsp.Schedule(d, 16, tsp.make_opts(flags=tsp.FLAG_INJECT_STALL)).validate()
    assert st == 0, why                                      # the hook acts only at upload


def test_waves_have_one_arrival_per_cta_and_phase():
    s = _sched("tiny", n=16, scheduler=0)
    tasks, off = s.tasks()
    per = {}
    for c in range(16):
        for i in range(off[c], off[c + 1]):
            t = tasks[i]
            key = (c, t.phase_kind, t.layer)
            per[key] = per.get(key, 0) + (t.signal_ctr != tsp.NO_COUNTER)
    assert set(per.values()) == {1}
