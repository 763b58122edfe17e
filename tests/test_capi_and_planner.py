"""C ABI exports and the planner/validator, on the CPU (no GPU calls)."""
import ctypes
import os
import re

import numpy as np
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


# ------------------------------------------------------------------ chunk geometry
def _ceil(a, b):
    return -(-a // b)


def _chain_budget(cfg, wb, kv8=False, slot_bytes=0):
    """The chunk budget of the chain's GEMVs (Q/K/V, O-projection) and of a BF16
    KV block: the caller's slot, else 16 KB, four hidden-wide rows or the
    longest row (two for gate/up), whichever is largest, in whole KB."""
    if slot_bytes:
        return slot_bytes
    H, F, qd, d = cfg.hidden, cfg.ffn, cfg.q_dim, cfg.head_dim
    need = max(wb * H, wb * qd, wb * F, 2 * wb * H, 2 * 8192 + 2 * (8192 // d) * 4 if kv8 else 0)
    return _ceil(max(need, 16384, 4 * wb * H), 1024) * 1024


def _check_slot_growth(info, cfg, wb, n, chain, grows):
    """The slot is the chain budget, or, for a default plan (`grows`), the
    largest whole number k of gate/up pairs above it with eight slots within
    227 KB of shared memory and k <= ceil(F / CTAs) / 16 (two ring laps)."""
    slot, pair = info["slot_bytes"], 2 * wb * cfg.hidden
    rest = info["smem_bytes"] - info["ring_slots"] * slot   # control block + vector area
    kmax = _ceil(cfg.ffn, n) // 16 if grows else 0
    fits = [k for k in range(kmax, 0, -1)
            if _ceil(k * pair, 1024) * 1024 > chain and rest + 8 * _ceil(k * pair, 1024) * 1024 <= 232448]
    # the loop stops at the first k whose slot is not above the chain budget
    stop = next((k for k in range(kmax, 0, -1) if _ceil(k * pair, 1024) * 1024 <= chain), 0)
    fits = [k for k in fits if k > stop]
    want = _ceil(fits[0] * pair, 1024) * 1024 if fits else chain
    assert slot == want, (slot, want, chain)


def test_int8_layer_chunks_give_every_consumer_warp_work():
    """INT8 layer GEMVs: rows per chunk = min(what fills the op's budget (at
    most 8), ceil(ceil(rows / CTAs) / 8)); the LM head and BF16 keep full
    chunks. Q/K/V and the O-projection fill the chain budget, the rest the
    slot."""
    for name in ("llama1b", "qwen3_0_6b", "qwen3_4b"):
        cfg = S.CONFIGS[name]
        H, F, qkv = cfg.hidden, cfg.ffn, cfg.q_dim + 2 * cfg.kv_dim
        bi, qi = _sched(name).info(), _sched(name, weight_format=tsp.WEIGHTS_INT8).info()
        b, q = bi["rows_per_chunk"], qi["rows_per_chunk"]
        slot = {2: bi["slot_bytes"], 1: qi["slot_bytes"]}
        chain = {2: _chain_budget(cfg, 2), 1: _chain_budget(cfg, 1)}
        _check_slot_growth(bi, cfg, 2, 152, chain[2], True)
        _check_slot_growth(qi, cfg, 1, 152, chain[1], True)
        full = lambda width, mats, wb: min(8, slot[wb] // (width * wb * mats))
        cfull = lambda width, mats, wb: min(8, chain[wb] // (width * wb * mats))
        assert b == {"qkv": cfull(H, 1, 2), "o": cfull(cfg.q_dim, 1, 2), "gateup": full(H, 2, 2),
                     "down": full(F, 1, 2), "lm": full(H, 1, 2)}
        cap = lambda rows: _ceil(_ceil(rows, 152), 8)
        assert q == {"qkv": max(1, min(cfull(H, 1, 1), cap(qkv))),
                     "o": max(1, min(cfull(cfg.q_dim, 1, 1), cap(H))),
                     "gateup": max(1, min(full(H, 2, 1), cap(F))),
                     "down": max(1, min(full(F, 1, 1), cap(H))),
                     "lm": full(H, 1, 1)}
    # worked by hand for the Llama-1B shape: 3072 Q/K/V rows -> 21 per CTA -> 3 per chunk
    assert _sched("llama1b", weight_format=tsp.WEIGHTS_INT8).info()["rows_per_chunk"] == \
        {"qkv": 3, "o": 2, "gateup": 4, "down": 2, "lm": 8}


def test_default_slot_grows_by_whole_gate_up_pairs():
    """Worked by hand, 152 CTAs. Llama-1B shape, BF16: 54 gate/up pairs of
    8 KB per CTA allow at most 3 pairs a chunk (two laps of 8), and 8 x 24 KB
    fit, so 24 KB slots with 3 pairs, 6 LM-head rows, but Q/K/V and O at the
    16 KB budget (4 rows) and 64-position KV blocks. Qwen3-0.6B: 21 pairs
    allow 1 pair (4 KB), under 16 KB: no growth. Qwen3-4B BF16: 64 pairs of
    10 KB allow 4, but only 2 (20 KB, the budget itself) fit. Qwen3-4B INT8:
    4 pairs of 5 KB = 20 KB over a 16 KB budget. A slot or ring size given by
    the caller turns the growth off."""
    i = _sched("llama1b").info()
    assert (i["slot_bytes"], i["ring_slots"], i["kv_block"]) == (24576, 8, 64)
    assert i["rows_per_chunk"] == {"qkv": 4, "o": 4, "gateup": 3, "down": 1, "lm": 6}
    assert i["smem_bytes"] <= 232448
    assert _sched("llama1b", kv_format=tsp.KV_INT8).info()["slot_bytes"] == 24576
    assert _sched("qwen3_0_6b").info()["slot_bytes"] == 16384
    assert _sched("qwen3_4b").info()["slot_bytes"] == 20480
    q4 = _sched("qwen3_4b", weight_format=tsp.WEIGHTS_INT8).info()
    assert q4["slot_bytes"] == 20480 and q4["rows_per_chunk"]["gateup"] == 4
    assert _sched("llama1b", weight_format=tsp.WEIGHTS_INT8).info()["slot_bytes"] == 16384
    for opts in (dict(slot_bytes=16384), dict(ring_slots=8)):
        j = _sched("llama1b", **opts).info()
        assert j["slot_bytes"] == 16384
        assert j["rows_per_chunk"] == {"qkv": 4, "o": 4, "gateup": 2, "down": 1, "lm": 4}


def test_tensor_core_attention_only_where_a_split_can_reach_eight_chunks():
    """The owner form (one warp per chunk) only where a split can reach 8
    chunks: 1,088 positions in 64-position blocks over 17 splits: at most 1
    chunk per split (shared chunks); 32,832 positions over 19 splits: up to
    28."""
    short, long_ = _sched("llama1b").info(), _sched("llama1b_long").info()
    assert (short["kv_block"], short["kv_splits"], short["attn_tensor_cores"]) == (64, 17, 0)
    assert (long_["kv_block"], long_["kv_splits"], long_["attn_tensor_cores"]) == (64, 19, 1)
    # fewer splits turn it on for a short context too: 17 blocks over 2 splits -> 9 chunks
    assert _sched("llama1b", kv_splits=2).info()["attn_tensor_cores"] == 1
    assert _sched("llama1b", kv_splits=3).info()["attn_tensor_cores"] == 0      # 6 chunks
    # head_dim 128: 32-position blocks
    assert _sched("qwen3_4b").info()["kv_block"] == 32


def test_kv_block_is_capped_at_one_tma_box():
    """A 64 KB slot holds 256 positions of K and V at d = 64; 96 KB would hold
    384, more than a tensor-map box (256 rows): the chunk stays at 256."""
    d = tsp.ModelDesc.from_config(S.CONFIGS["tiny"])
    for slot, want in ((65536, 256), (98304, 256), (32768, 128)):
        s = tsp.Schedule(d, 16, tsp.make_opts(slot_bytes=slot, ring_slots=2))
        assert s.info()["kv_block"] == want
        assert s.validate()[0] == 0


def test_random_shapes_build_valid_schedules_with_consistent_chunk_geometry():
    """Seeded random decoders (head_dim, GQA group, widths, depth, context,
    CTA count, scheduler, weight format, splits): every schedule the planner
    builds validates, and its chunk geometry follows the rules the kernel
    relies on (rows per chunk >= 1 and within the slot; the INT8 cap; the
    tensor-core attention flag). Vocabularies smaller than the grid are
    included. Only documented rejections are allowed."""
    from dataclasses import replace
    rng = np.random.default_rng(51)
    built = 0
    for _ in range(200):
        d = int(rng.choice([64, 128]))
        nkv = int(rng.integers(1, 9))
        nq = nkv * int(rng.choice([1, 2, 4, 8]))
        cfg = replace(S.CONFIGS["tiny"], n_layers=int(rng.integers(1, 6)),
                      hidden=int(rng.integers(2, 48)) * 64, n_q_heads=nq, n_kv_heads=nkv,
                      head_dim=d, ffn=int(rng.integers(4, 120)) * 32,
                      vocab=int(rng.integers(100, 6000)), max_pos=int(rng.integers(16, 6000)),
                      qk_norm=bool(rng.integers(0, 2)))
        n = int(rng.choice([1, 7, 37, 152, int(rng.integers(1, 300))]))
        opts = dict(scheduler=int(rng.integers(0, 3)), weight_format=int(rng.integers(0, 2)))
        if rng.random() < 0.3:
            opts["kv_splits"] = int(rng.integers(1, 40))
        try:
            sch = tsp.Schedule(tsp.ModelDesc.from_config(cfg), n, tsp.make_opts(**opts))
        except tsp.TilesError as e:
            assert e.status in (-1, -2), e.status             # bad option / unsupported shape
            continue
        st, why = sch.validate()
        assert st == 0, why
        info = sch.info()
        wb = 1 if opts["weight_format"] == tsp.WEIGHTS_INT8 else 2
        H, F, qd = cfg.hidden, cfg.ffn, cfg.q_dim
        qkv = qd + 2 * cfg.kv_dim
        slot = info["slot_bytes"]
        chain = _chain_budget(cfg, wb, opts.get("kv_format", 0) == tsp.KV_INT8, opts.get("slot_bytes", 0))
        _check_slot_growth(info, cfg, wb, n, chain, "slot_bytes" not in opts and "ring_slots" not in opts)
        widths = {"qkv": (H, 1, qkv), "o": (qd, 1, H), "gateup": (H, 2, F), "down": (F, 1, H),
                  "lm": (H, 1, 0)}
        for op, rows in info["rows_per_chunk"].items():
            width, mats, out_rows = widths[op]
            full = min(8, (chain if op in ("qkv", "o") else slot) // (width * wb * mats))
            assert 1 <= rows <= full and rows * width * wb * mats <= slot
            if wb == 1 and op != "lm":
                assert rows == max(1, min(full, _ceil(_ceil(out_rows, n), 8)))
            else:
                assert rows == full
        kvb, S_ = info["kv_block"], info["kv_splits"]
        assert 16 <= kvb <= 256 and kvb % 16 == 0 and 2 * kvb * d * 2 <= chain
        want = _ceil(_ceil(cfg.max_pos, kvb), S_) >= 8 and kvb % (2048 // d) == 0
        assert info["attn_tensor_cores"] == int(want)
        built += 1
    assert built >= 120


def test_small_vocabulary_confines_attention_to_lm_head_ctas():
    """A vocabulary with fewer rows than CTAs (107 rows on 152 CTAs, more
    attention items per layer than rows): under tag-carrying activations every
    CTA with attention work must signal the LM head ("Tiles: Scheduling LLM
    Decoding as a Graph of Tiles", What the code contains: the schedule is
    validated before launch). The planner confines every layer's attention
    items to 107 CTAs, one LM-head row each, and all three schedulers
    validate. With a vocabulary of at least one row per CTA the attention
    items are unrestricted."""
    from dataclasses import replace
    cfg = replace(S.CONFIGS["tiny"], vocab=107, n_layers=4)
    for sched in (tsp.SCHED_FLAGS, tsp.SCHED_COUNTERS, tsp.SCHED_WAVES):
        sch = tsp.Schedule(tsp.ModelDesc.from_config(cfg), 152, tsp.make_opts(scheduler=sched, kv_splits=64))
        st, why = sch.validate()
        assert st == 0, why
        tasks, off = sch.tasks()
        attn, lm = set(), {}
        for c in range(152):
            for i in range(off[c], off[c + 1]):
                t = tasks[i]
                if t.op == 2:
                    attn.add(c)
                elif t.op == 7:
                    lm[c] = lm.get(c, 0) + (t.end - t.begin)
        assert sum(lm.values()) == 107 and len(lm) == 107
        assert attn <= set(lm), sorted(attn - set(lm))
        assert len(attn) > 64          # 2 KV heads x 64 splits per layer spread over 107 CTAs
    big = replace(cfg, vocab=1024)
    sch = tsp.Schedule(tsp.ModelDesc.from_config(big), 152, tsp.make_opts(kv_splits=64))
    tasks, off = sch.tasks()
    attn = {c for c in range(152) for i in range(off[c], off[c + 1]) if tasks[i].op == 2}
    assert len(attn) == 152


def test_int8_kv_layout_and_schedule_geometry():
    """The INT8 KV cache ("History and roadmap", M8: INT8 KV cache with
    smoothed keys): buffer layout (position stride rounded up to 16, parts at
    256-byte offsets), the chunk geometry the kernel relies on (8 KB of key
    codes and 8 KB of value codes per chunk plus their scales, in one slot;
    every split on the tensor-core form), and the streamed bytes the planner
    balances: 2 d + 8 bytes per cached position and head instead of 4 d."""
    from dataclasses import replace
    for d, nkv, L, mp in ((64, 8, 16, 32832), (128, 8, 28, 1088), (64, 2, 2, 130)):
        cfg = replace(S.CONFIGS["tiny"], head_dim=d, n_kv_heads=nkv, n_q_heads=nkv * 2, n_layers=L, max_pos=mp)
        lay = tsp.kv8_layout(tsp.ModelDesc.from_config(cfg))
        Z, MP = L * nkv, _ceil(mp, 16) * 16
        assert lay["pos_stride"] == MP
        assert lay["k_scale_off"] == _ceil(Z * MP * d, 256) * 256
        assert lay["k_mu_off"] == _ceil(lay["k_scale_off"] + Z * MP * 4, 256) * 256
        assert lay["k_bytes"] == lay["k_mu_off"] + Z * d * 4
        assert lay["v_scale_off"] == _ceil(Z * d * MP, 256) * 256
        assert lay["v_bytes"] == lay["v_scale_off"] + Z * MP * 4
        sch = tsp.Schedule(tsp.ModelDesc.from_config(cfg), 152, tsp.make_opts(kv_format=tsp.KV_INT8))
        assert sch.validate()[0] == 0
        info = sch.info()
        assert info["kv_format"] == tsp.KV_INT8 and info["attn_tensor_cores"] == 1
        assert info["kv_block"] == 8192 // d
        assert info["slot_bytes"] >= 2 * 8192 + 2 * (8192 // d) * 4 and info["slot_bytes"] % 1024 == 0
    # streamed bytes at a long context: weights the same, K/V at (2d + 8) / 4d
    cfg = S.CONFIGS["llama1b_long"]
    desc = tsp.ModelDesc.from_config(cfg)
    b16 = tsp.Schedule(desc, 152, tsp.make_opts())
    b8 = tsp.Schedule(desc, 152, tsp.make_opts(kv_format=tsp.KV_INT8))
    P = cfg.start_pos
    w = b16.info()["weight_bytes_per_token"]
    assert b8.info()["weight_bytes_per_token"] == w
    kv16, kv8 = sum(b16.cta_bytes(P)) - w, sum(b8.cta_bytes(P)) - w
    per_pos = cfg.n_layers * cfg.n_kv_heads
    assert kv16 == per_pos * P * 4 * cfg.head_dim
    assert kv8 == per_pos * P * (2 * cfg.head_dim + 8)
    with pytest.raises(tsp.TilesError):
        tsp.Schedule(desc, 152, tsp.make_opts(kv_format=2))
