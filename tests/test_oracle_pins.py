"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each oracle function is checked against something other than itself: values
the pages print (fixtures under tests/golden/, each citing its passage),
closed forms, invariants, library routines that compute the same thing, and
brute force on tiny inputs.  Pages cited:
  a2a-backends  vincentzed.com/writing/a2a-backends
  Beyond One GPU  ishwarj.com/writings/llm-inference-7-beyond-one-gpu
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import moe_synth as ms
import oracle

MiB = 1024 * 1024


def _golden(name):
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ bf16 --

def test_bf16_round_trip_and_ties():
    # exact values survive; halfway cases go to the even neighbour
    for b in (0x0000, 0x8000, 0x3F80, 0xBF80, 0x7F7F, 0x0001, 0x8001, 0x4049):
        assert oracle.bf16_from_double(oracle.bf16_to_double(b)) == b
    one = 1.0
    ulp = 2.0 ** -7
    assert oracle.bf16_from_double(one + ulp / 2) == 0x3F80          # tie -> even (1.0)
    assert oracle.bf16_from_double(one + 3 * ulp / 2) == 0x3F82      # tie -> even (1 + 2ulp)
    assert oracle.bf16_from_double(one + ulp / 2 + 2 ** -40) == 0x3F81  # just above the tie
    assert oracle.bf16_from_double(-(one + ulp / 2)) == 0xBF80
    assert oracle.bf16_from_double(3.0e38 * 2) == 0x7F80             # overflow -> inf
    assert oracle.bf16_from_double(2.0 ** -134) == 0x0000            # below half the smallest subnormal
    assert oracle.bf16_from_double(3 * 2.0 ** -134) == 0x0002        # 1.5 quanta -> even (2 quanta)


def test_bf16_matches_bit_trick_on_floats():
    # For float32-representable inputs a single rounding to bf16 equals the
    # classic add-0x7FFF-plus-lsb bit trick (an independent formulation).
    rng = np.random.default_rng(1)
    f = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    want = ms.bf16_bits_from_f32(f)
    got = np.array([oracle.bf16_from_double(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_double_rounding_is_avoided():
    # 1 + 2^-8 + 2^-30 is above the halfway point: one rounding gives 1 + 2^-7,
    # while rounding to float32 first (1 + 2^-8, a tie) then to bf16 gives 1.0.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert oracle.bf16_from_double(v) == 0x3F81


# ------------------------------------------- copies per token, a2a-backends 1.3 --

def test_expected_copies_printed_values():
    g = _golden("copies_closed_form.json")
    for c in g["cases"]:
        v = oracle.expected_copies(c["E"], c["G"], c["k"])
        assert round(v, g["printed_decimals"]) == pytest.approx(c["printed"], abs=1e-9), c


@pytest.mark.parametrize("E,G,k", [(8, 4, 3), (12, 3, 4), (9, 3, 2), (10, 5, 1), (8, 2, 8)])
def test_expected_copies_brute_force(E, G, k):
    # average over every k-subset of the number of blocks it touches
    L = E // G
    tot = 0
    n = 0
    for sub in itertools.combinations(range(E), k):
        tot += len({e // L for e in sub})
        n += 1
    assert oracle.expected_copies(E, G, k) == pytest.approx(tot / n, rel=1e-12)


# -------------------------------------------------------- route (a2a 1.1) --

def _check_topk(logits, ids, w, k):
    E = logits.shape[-1]
    for n in range(logits.shape[0]):
        row = logits[n]
        sel = ids[n]
        assert len(set(sel.tolist())) == k
        unsel = np.setdiff1d(np.arange(E), sel)
        # every chosen logit >= every other one; equal ones resolved to the lower id
        if unsel.size:
            m_un = row[unsel].max()
            assert row[sel].min() >= m_un
            for e in sel:
                for e2 in unsel:
                    if row[e] == row[e2]:
                        assert e < e2
        # descending order, ties by ascending id
        for a, b in zip(sel[:-1], sel[1:]):
            assert row[a] > row[b] or (row[a] == row[b] and a < b)
        # weights: positive, sum to one, ratios are exp of logit differences
        assert np.all(w[n] > 0)
        assert w[n].sum() == pytest.approx(1.0, abs=1e-12)
        for j in range(k):
            assert w[n, j] / w[n, 0] == pytest.approx(math.exp(float(row[sel[j]]) - float(row[sel[0]])),
                                                      rel=1e-12)


def test_route_topk_properties_random():
    w_ = ms.workload("tiny")
    logits = ms.gen_logits(w_)[0]
    ids, w = oracle.route_topk(logits, w_.k)
    _check_topk(logits, ids, w, w_.k)


def test_route_topk_ties_pick_lower_id():
    rng = np.random.default_rng(7)
    logits = rng.integers(-2, 3, size=(64, 10)).astype(np.float32)  # many ties
    ids, w = oracle.route_topk(logits, 4)
    _check_topk(logits, ids, w, 4)
    # all-equal row: the k lowest ids, equal weights
    ids, w = oracle.route_topk(np.zeros((1, 7), np.float32), 3)
    assert ids.tolist() == [[0, 1, 2]]
    assert np.allclose(w, 1 / 3)


def test_route_topk_full_softmax_and_k1():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((20, 12)).astype(np.float32)
    ids, w = oracle.route_topk(logits, 12)  # k = E: plain softmax, reordered
    for n in range(20):
        ref = scipy_special.softmax(logits[n].astype(np.float64))
        assert np.allclose(w[n], ref[ids[n]], rtol=1e-12, atol=0)
        assert np.array_equal(ids[n], np.argsort(-logits[n].astype(np.float64), kind="stable"))
    ids, w = oracle.route_topk(logits, 1)  # k = 1: argmax with weight 1
    assert np.array_equal(ids[:, 0], np.argmax(logits, axis=1))
    assert np.all(w == 1.0)


def test_route_topk_brute_force_subsets():
    # the chosen set maximises the sum of logits over all k-subsets (distinct logits)
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((30, 7)).astype(np.float32)
    k = 3
    ids, _ = oracle.route_topk(logits, k)
    for n in range(30):
        best = max(itertools.combinations(range(7), k), key=lambda s: sum(float(logits[n, e]) for e in s))
        assert set(ids[n].tolist()) == set(best)


# ---------------------------------------------------- layout (a2a 1.1, 1.3, 3.2) --

def test_layout_fig1_two_copies():
    g = _golden("fig1_two_copies.json")
    ids = np.array(g["ids"], np.int32)[None]
    lay = oracle.dispatch_layout(ids, g["E"], g["P"])
    assert int(lay["part_offsets"][0, -1]) == g["expected_copies"]
    hit = [p for p in range(g["P"]) if lay["token_slot"][0, 0, p] >= 0]
    assert hit == g["expected_partitions"]
    assert int(lay["expert_counts"].sum()) == 3


def _brute_layout(ids, E, P):
    """Independent formulation: list every (partition, token) pair a token needs,
    sort the list by (partition, token) and number it 0, 1, 2, ...; for expert
    ranks, number each expert's pairs by sorting their (token, slot) positions."""
    S, T, k = ids.shape
    L = E // P
    slot = -np.ones((S, T, P), np.int64)
    counts = np.zeros((S, P), np.int64)
    ecounts = np.zeros((S, E), np.int64)
    rank = -np.ones((S, T, k), np.int64)
    for s in range(S):
        need = sorted({(int(e) // L, t) for t in range(T) for e in ids[s, t] if 0 <= e < E})
        for i, (p, t) in enumerate(need):
            slot[s, t, p] = i
            counts[s, p] += 1
        for e in ids[s].ravel():
            if 0 <= e < E:
                ecounts[s, e] += 1
        for e in range(E):
            where = sorted((t, j) for t in range(T) for j in range(k) if ids[s, t, j] == e)
            for r, (t, j) in enumerate(where):
                rank[s, t, j] = r
    return slot, counts, ecounts, rank


def test_layout_brute_force_all_tiny_inputs():
    # every id assignment of T=2 tokens, k=2, E=4 (ids in -1..4, 4 = out of range), P=2
    E, P, k, T = 4, 2, 2, 2
    vals = [-1, 0, 1, 2, 3, 4]
    for combo in itertools.product(vals, repeat=T * k):
        ids = np.array(combo, np.int32).reshape(1, T, k)
        lay = oracle.dispatch_layout(ids, E, P)
        slot, counts, ecounts, rank = _brute_layout(ids, E, P)
        assert np.array_equal(lay["token_slot"], slot), combo
        assert np.array_equal(lay["part_counts"], counts), combo
        assert np.array_equal(lay["expert_counts"], ecounts), combo
        assert np.array_equal(lay["expert_rank"], rank), combo
        assert np.array_equal(lay["part_offsets"][:, 1:], np.cumsum(counts, axis=1)), combo
        assert (lay["status"] == oracle.BIT_BAD_ID) == (4 in combo), combo


def test_layout_brute_force_random_small():
    rng = np.random.default_rng(5)
    for _ in range(40):
        S, T, P = int(rng.integers(1, 3)), int(rng.integers(0, 9)), int(rng.integers(1, 5))
        L = int(rng.integers(1, 3))
        E = P * L
        k = int(rng.integers(1, min(E, 3) + 1))
        ids = rng.integers(-1, E, size=(S, T, k)).astype(np.int32)
        lay = oracle.dispatch_layout(ids, E, P)
        slot, counts, ecounts, rank = _brute_layout(ids, E, P)
        assert np.array_equal(lay["token_slot"], slot)
        assert np.array_equal(lay["part_counts"], counts)
        assert np.array_equal(lay["expert_counts"], ecounts)
        assert np.array_equal(lay["expert_rank"], rank)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "large"])
def test_layout_invariants(name):
    w_ = ms.workload(name)
    ids, _ = oracle.route_topk(ms.gen_logits(w_), w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    S, T = w_.S, w_.T
    assert lay["status"] == 0
    assert lay["expert_counts"].sum() == S * T * w_.k            # nothing skipped
    copies = (lay["token_slot"] >= 0).sum(axis=2)
    assert copies.min() >= 1 and copies.max() <= min(w_.k, w_.P)
    assert np.array_equal(lay["part_offsets"][:, -1], copies.sum(axis=1))
    for s in range(S):
        for p in range(w_.P):
            sl = lay["token_slot"][s, :, p]
            v = sl[sl >= 0]
            lo, hi = lay["part_offsets"][s, p], lay["part_offsets"][s, p + 1]
            assert np.array_equal(v, np.arange(lo, hi))                 # dense, ascending in t
        # each expert's ranks, read in stable-sort order of its pairs, are 0, 1, 2, ...
        flat = ids[s].reshape(-1)
        order = np.argsort(flat, kind="stable")
        rk = lay["expert_rank"][s].reshape(-1)[order]
        starts = np.concatenate([[0], np.cumsum(lay["expert_counts"][s])[:-1]])
        want = np.arange(flat.size) - np.repeat(starts, lay["expert_counts"][s])
        assert np.array_equal(rk, want)


def _mean_copies_sigma(E, P, k, T):
    """Standard error of the mean copy count under uniform routing (exact variance)."""
    L = E // P
    q1 = math.comb(E - L, k) / math.comb(E, k)           # P(partition missed)
    q2 = math.comb(E - 2 * L, k) / math.comb(E, k)       # P(two given partitions missed)
    var = P * q1 * (1 - q1) + P * (P - 1) * (q2 - q1 * q1)
    return math.sqrt(var / T)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "large"])
def test_mean_copies_matches_closed_form(name):
    w_ = ms.workload(name)
    ids, _ = oracle.route_topk(ms.gen_logits(w_), w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    c = lay["part_offsets"][0, -1] / w_.T
    mu = oracle.expected_copies(w_.E, w_.P, w_.k)
    sig = _mean_copies_sigma(w_.E, w_.P, w_.k, w_.T)
    assert abs(c - mu) < 5 * sig, (c, mu, sig)


def test_bytes_per_gpu_printed_values():
    g = _golden("bytes_per_gpu.json")
    rb = g["row_bytes"]
    for case in g["cases"]:
        T = case["rows_per_gpu"]
        w_ = ms.workload("prefill", T=T) if T == 4096 else ms.workload("decode", T=T)
        ids, _ = oracle.route_topk(ms.gen_logits(w_), w_.k)
        lay = oracle.dispatch_layout(ids, g["E"], g["G"])
        broadcast = g["G"] * T * rb / MiB
        per_expert = lay["expert_counts"].sum() * rb / MiB
        dedup = lay["part_offsets"][0, -1] * rb / MiB
        assert broadcast == pytest.approx(case["broadcast_MiB"], abs=0.05)
        assert per_expert == pytest.approx(case["per_expert_MiB"], abs=0.05)
        # sampled copies: 5 standard errors of the mean, plus the page's rounding
        sig = _mean_copies_sigma(g["E"], g["G"], g["k"], T) * T * rb / MiB
        half_digit = 0.5 if case["dedup_MiB"] >= 100 else 0.05
        assert abs(dedup - case["dedup_MiB"]) <= 5 * sig + half_digit, (dedup, sig)
        # the closed-form expectation itself reproduces the printed figure
        mu = oracle.expected_copies(g["E"], g["G"], g["k"]) * T * rb / MiB
        assert abs(mu - case["dedup_MiB"]) <= half_digit


def test_byte_model_per_expert_copies():
    g = _golden("byte_model_b1g.json")
    assert g["k"] * g["d"] * (g["s_dispatch"] + g["s_combine"]) == g["bytes_per_token"]
    # the oracle's per-expert count (sum of expert_counts) gives one copy per chosen expert
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((1, g["tokens"], g["E"])).astype(np.float32)
    ids, _ = oracle.route_topk(logits, g["k"])
    lay = oracle.dispatch_layout(ids, g["E"], 8)
    mb = lay["expert_counts"].sum() * g["d"] * g["s_dispatch"] / 1e6
    assert round(mb, 2) == g["dispatch_MB_1e6"]


# ------------------------------------------------------------- pack (a2a 3.2) --

def test_pack_rows_are_bit_copies():
    w_ = ms.workload("tiny")
    inp = ms.gen_inputs(w_)
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap = w_.T * min(w_.k, w_.P)
    send, src, st = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap)
    assert st == 0
    used = lay["part_offsets"][0, -1]
    assert np.all(src[0, :used] >= 0) and np.all(src[0, used:] == -1)
    assert np.array_equal(send[0, :used], inp["x"][0, src[0, :used]])
    for p in range(w_.P):
        seg = src[0, lay["part_offsets"][0, p]:lay["part_offsets"][0, p + 1]]
        assert np.all(np.diff(seg) > 0)                                   # ascending tokens
        # exactly the tokens that need partition p
        need = [t for t in range(w_.T) if any(e // (w_.E // w_.P) == p for e in ids[0, t])]
        assert seg.tolist() == need


def test_pack_capacity_drop():
    w_ = ms.workload("tiny")
    inp = ms.gen_inputs(w_)
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap = 100
    send, src, st = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap)
    assert st == oracle.BIT_CAPACITY
    assert np.all(src[0] >= 0)
    assert np.array_equal(send[0], inp["x"][0, src[0]])


# --------------------------------------------------- permute (a2a 1.5, 3.3, 5.1) --

def test_permute_regroup_5_to_7():
    g = _golden("regroup_5_to_7.json")
    ids = np.array(g["ids"], np.int32)[None]
    T = ids.shape[1]
    H = 8
    x = np.arange(T * H, dtype=np.uint16).reshape(1, T, H) + 1
    lay = oracle.dispatch_layout(ids, g["E"], g["P"])
    p = g["recv_part"]
    assert lay["part_counts"][0, p] == g["expected_arrived_rows"]
    send, src, _ = oracle.dispatch_pack(x, lay["token_slot"], T * 2)
    per = oracle.permute_to_experts(send, lay["token_slot"], ids, g["E"], recv_part=p)
    off = per["expert_offsets"]
    assert off[-1] == g["expected_permuted_rows"]
    for e_str, toks in g["expected_expert_runs"].items():
        e = int(e_str)
        rows = per["recv"][off[e]:off[e + 1]]
        assert np.array_equal(rows, x[0, toks])
    assert np.all(per["pair_row"][0][ids[0] // 4 != p] == -1)


def _stable_sort_pin(ids, recv_part, E, P, per):
    """The permuted order is a stable sort of the receiving pairs by expert id."""
    flat = ids.reshape(-1)
    L = E // P
    q = np.nonzero((flat >= 0) & (flat < E) & ((recv_part < 0) | (flat // L == recv_part)))[0]
    order = q[np.argsort(flat[q], kind="stable")]
    rp = per["recv_pair"]
    got = rp[rp >= 0]
    assert np.array_equal(got, order)


@pytest.mark.parametrize("name,align,recv_part", [("tiny", 1, -1), ("tiny", 128, -1), ("tiny", 8, 2),
                                                  ("decode", 1, -1), ("decode", 128, 3)])
def test_permute_stable_sort_and_inverse(name, align, recv_part):
    w_ = ms.workload(name)
    inp = ms.gen_inputs(w_)
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap = w_.T * min(w_.k, w_.P)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap)
    per = oracle.permute_to_experts(send, lay["token_slot"], ids, w_.E, recv_part=recv_part, align=align)
    assert per["status"] == 0
    _stable_sort_pin(ids, recv_part, w_.E, w_.P, per)
    pr = per["pair_row"].reshape(-1)
    rp = per["recv_pair"]
    valid = np.nonzero(pr >= 0)[0]
    assert np.array_equal(rp[pr[valid]], valid)                  # recv_pair o pair_row = id
    rows = np.nonzero(rp >= 0)[0]
    assert np.array_equal(pr[rp[rows]], rows)                    # pair_row o recv_pair = id
    off = per["expert_offsets"]
    assert np.all(np.diff(off) % align == 0)
    L = w_.E // w_.P
    for e in range(w_.E):
        rr = np.arange(off[e], off[e + 1])
        real = rr[rp[rr] >= 0]
        pad = rr[rp[rr] < 0]
        assert np.all(ids.reshape(-1)[rp[real]] == e)
        assert np.all(per["recv"][pad] == 0)
        if recv_part >= 0 and e // L != recv_part:
            assert rr.size == 0
    # each row is the source token's row
    tok = rows // w_.k
    assert np.array_equal(per["recv"][rows], inp["x"].reshape(-1, w_.H)[rp[rows] // w_.k])
    _ = tok


def test_permute_capacity_drop_and_bad_id():
    w_ = ms.workload("tiny")
    inp = ms.gen_inputs(w_)
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    ids = ids.copy()
    ids[0, 5, 1] = w_.E + 3      # out of range: skipped and flagged
    ids[0, 6, 0] = -1            # not routed: skipped silently
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    assert lay["status"] == oracle.BIT_BAD_ID
    cap = w_.T * min(w_.k, w_.P)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap)
    per = oracle.permute_to_experts(send, lay["token_slot"], ids, w_.E, cap_recv=100)
    assert per["status"] == (oracle.BIT_BAD_ID | oracle.BIT_CAPACITY)
    pr = per["pair_row"].reshape(-1)
    assert pr.max() < 100 and (pr >= 0).sum() == 100
    assert pr[5 * w_.k + 1] == -1 and pr[6 * w_.k + 0] == -1


# ------------------------------------------------------------ combine (a2a 7.1) --

@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_identity_round_trip(name):
    # identity experts and weights that sum to one return the input rows
    w_ = ms.workload(name)
    inp = ms.gen_inputs(w_)
    r = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, ms.gen_scales(w_, identity=True))
    assert np.array_equal(r["out"], inp["x"])


def test_identity_round_trip_with_alignment():
    w_ = ms.workload("tiny")
    inp = ms.gen_inputs(w_)
    r = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, None, align=128)
    assert np.array_equal(r["out"], inp["x"])


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_combine_closed_form_for_scalar_experts(name):
    # every pair of a token carries the same row x, so out = x * sum_j w_j s_{e_j}
    w_ = ms.workload(name)
    inp = ms.gen_inputs(w_)
    r = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, inp["scales"])
    ids = r["ids"]
    w32 = r["w"].astype(np.float32).astype(np.float64)
    factor = (w32 * inp["scales"].astype(np.float64)[ids]).sum(axis=2)          # [S, T]
    ref = ms.f32_from_bf16_bits(inp["x"]).astype(np.float64) * factor[..., None]
    got = ms.f32_from_bf16_bits(r["out"]).astype(np.float64)
    # two bf16 roundings (expert output, final sum): 2^-8 relative each
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30)


def test_combine_partials_sum_to_full():
    # stage-1 partial combines over each receiving partition add up to the full combine (a2a 7.1)
    w_ = ms.workload("tiny")
    inp = ms.gen_inputs(w_)
    full = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, inp["scales"])
    acc = np.zeros(inp["x"].shape, np.float64)
    for p in range(w_.P):
        part = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, inp["scales"], recv_part=p)
        acc += ms.f32_from_bf16_bits(part["out"])
    ref = ms.f32_from_bf16_bits(full["out"]).astype(np.float64)
    assert np.all(np.abs(acc - ref) <= 1e-2 * np.maximum(np.abs(ref), 1e-3))


def test_combine_skips_invalid_pairs_and_empty_tokens():
    H = 16
    y = ms.bf16_bits_from_f32(np.arange(3 * H, dtype=np.float32).reshape(3, H) / 8)
    pair_row = np.array([[[0, -1], [-1, -1], [2, 1]]], np.int32)
    w = np.array([[[0.5, 0.25], [0.3, 0.7], [0.25, 0.75]]], np.float32)
    out = oracle.combine(y, pair_row, w)
    yf = ms.f32_from_bf16_bits(y).astype(np.float64)
    assert np.array_equal(out[0, 0], ms.bf16_bits_from_f32((0.5 * yf[0]).astype(np.float32)))
    assert np.all(out[0, 1] == 0)
    assert np.array_equal(out[0, 2], ms.bf16_bits_from_f32((0.25 * yf[2] + 0.75 * yf[1]).astype(np.float32)))


def test_expert_scale_exact_products():
    # tiny scales (e+1)/16 times bf16 values are exact in float32, so the
    # oracle's single rounding must equal float32 multiply + bit-trick rounding
    w_ = ms.workload("tiny")
    inp = ms.gen_inputs(w_)
    r = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, inp["scales"])
    per = r["permute"]
    off = per["expert_offsets"]
    for e in range(w_.E):
        rows = per["recv"][off[e]:off[e + 1]]
        want = ms.bf16_bits_from_f32(ms.f32_from_bf16_bits(rows) * np.float32(inp["scales"][e]))
        assert np.array_equal(r["y"][off[e]:off[e + 1]], want)


# ------------------------------------------------- masked layout (a2a 4.1, 4.2) --

def _decode_from_8_sources(seed_index=11):
    w_ = ms.workload("decode", S=8, index=seed_index)
    inp = ms.gen_inputs(w_)
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap_send = w_.T * min(w_.k, w_.P)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    return w_, inp, ids, lay, send


def test_masked_shape_and_mean_rows():
    g = _golden("masked_rows.json")
    w_, inp, ids, lay, send = _decode_from_8_sources()
    assert (w_.E // w_.P, w_.S, w_.T) == (g["local_experts"], g["gpus"], g["decode_rows_per_gpu"])
    block = g["gpus"] * g["cap"]
    total = 0
    for p in range(w_.P):
        per = oracle.permute_masked(send, lay["token_slot"], ids, w_.E, p, block)
        assert per["recv"].shape[0] == g["rows"]                 # 48 x 8 x 128 rows of room
        assert per["status"] == 0
        total += int(per["masked_counts"].sum())
    # every pair lands on exactly one receiver: the mean over receivers is S*T*k/P = 384
    assert total / w_.P == g["arriving_rows_mean"]


@pytest.mark.parametrize("recv_part", [0, 5, -1])
def test_masked_equals_contiguous_runs(recv_part):
    w_, inp, ids, lay, send = _decode_from_8_sources()
    block = 1024
    m_ = oracle.permute_masked(send, lay["token_slot"], ids, w_.E, recv_part, block)
    c_ = oracle.permute_to_experts(send, lay["token_slot"], ids, w_.E, recv_part=recv_part)
    L = w_.E // w_.P
    e0 = 0 if recv_part < 0 else recv_part * L
    off = c_["expert_offsets"]
    for b in range(m_["masked_counts"].size):
        e = e0 + b
        n = int(m_["masked_counts"][b])
        assert n == off[e + 1] - off[e]
        rows = slice(b * block, b * block + n)
        assert np.array_equal(m_["recv"][rows], c_["recv"][off[e]:off[e + 1]])
        assert np.array_equal(m_["recv_pair"][rows], c_["recv_pair"][off[e]:off[e + 1]])
        assert np.all(m_["recv_pair"][b * block + n:(b + 1) * block] == -1)
    valid = c_["pair_row"] >= 0
    assert np.array_equal(m_["pair_row"] >= 0, valid)


def test_masked_overflow_keeps_first_pairs():
    w_, inp, ids, lay, send = _decode_from_8_sources()
    block = 4
    per = oracle.permute_masked(send, lay["token_slot"], ids, w_.E, 2, block)
    assert per["status"] == oracle.BIT_CAPACITY
    L = w_.E // w_.P
    flat = ids.reshape(-1)
    for b in range(L):
        e = 2 * L + b
        q = np.nonzero(flat == e)[0]                # pairs of e in (s, t, j) order
        keep = q[:block]
        assert per["masked_counts"][b] == keep.size
        assert np.array_equal(per["recv_pair"][b * block:b * block + keep.size], keep)
        assert np.all(per["pair_row"].reshape(-1)[q[block:]] == -1)


# ------------------------------------------------ two-stage combine (a2a 7.1) --

def _staged(name, scales_identity=False, S=None):
    w_ = ms.workload(name) if S is None else ms.workload(name, S=S)
    inp = ms.gen_inputs(w_)
    sc = ms.gen_scales(w_, identity=scales_identity)
    r = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, sc)
    cap_send = w_.T * min(w_.k, w_.P)
    w32 = r["w"].astype(np.float32)
    ret, st1 = oracle.combine_stage1(r["y"], r["permute"]["pair_row"], w32, r["ids"],
                                     r["layout"]["token_slot"], w_.E, cap_send)
    out, st2 = oracle.combine_stage2(ret, r["layout"]["token_slot"])
    return w_, inp, r, ret, out, st1 | st2


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_two_stage_matches_single_stage(name):
    w_, inp, r, ret, out, st = _staged(name)
    assert st == 0
    ref = ms.f32_from_bf16_bits(r["out"]).astype(np.float64)
    got = ms.f32_from_bf16_bits(out).astype(np.float64)
    # one extra bf16 rounding per partial row (at most min(k, P) of them)
    assert np.all(np.abs(got - ref) <= 2.0 ** -6 * np.maximum(np.abs(ref), 1e-3))


def test_two_stage_returns_one_row_per_copy():
    # a2a 7.1: each way returns as many rows as it sent (one per destination partition)
    w_, inp, r, ret, out, st = _staged("tiny", S=2)
    lay = r["layout"]
    for s in range(w_.S):
        used = int(lay["part_offsets"][s, -1])
        slots = lay["token_slot"][s]
        assert (slots >= 0).sum() == used
        # every used return row is the pre-added sum of that partition's experts
        L = w_.E // w_.P
        t, p = 5, int(np.nonzero(slots[5] >= 0)[0][0])
        row = ret[s, slots[t, p]]
        ids = r["ids"][s, t]
        pr = r["permute"]["pair_row"][s, t]
        wt = r["w"][s, t].astype(np.float32).astype(np.float64)
        acc = sum(wt[j] * ms.f32_from_bf16_bits(r["y"][pr[j]]).astype(np.float64)
                  for j in range(w_.k) if ids[j] // L == p)
        # rounded once from double (the bf16 rounding itself is pinned above)
        want = np.array([oracle.bf16_from_double(float(v)) for v in acc], np.uint16)
        assert np.array_equal(row, want)


def test_two_stage_identity_round_trip_close():
    w_, inp, r, ret, out, st = _staged("decode", scales_identity=True)
    x = ms.f32_from_bf16_bits(inp["x"]).astype(np.float64)
    got = ms.f32_from_bf16_bits(out).astype(np.float64)
    assert np.all(np.abs(got - x) <= 2.0 ** -6 * np.maximum(np.abs(x), 1e-3))


# ---------------------------------------------- FP8 dispatch rows (a2a 7.2) --

def test_quantized_row_sizes():
    g = _golden("quantized_row_bytes.json")
    H = g["hidden"]
    assert 2 * H == g["bf16_bytes"]
    x = ms.gen_x(ms.workload("prefill"), T=1)[0, 0]
    codes, scales = oracle.quantize_mxfp8(x)
    assert codes.nbytes + scales.nbytes == g["fp8_bytes"]              # MXFP8: 1 B per 32
    assert H + H // g["deepep_v1_block"] * g["deepep_v1_scale_bytes"] == g["fp8_bytes"]
    assert H // 2 + H // g["nvfp4_block"] == g["nvfp4_bytes"]
    # one packed record per (token, partition) is exactly the page's FP8 row
    ts = np.zeros((1, 1, 1), np.int32)
    q, src, st = oracle.dispatch_pack_mxfp8(ms.gen_x(ms.workload("prefill"), T=1), ts, 1)
    assert q.shape == (1, 1, g["fp8_bytes"]) and st == 0 and src[0, 0] == 0


def test_e4m3_matches_torch_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(21)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-9, 6, 20000))).astype(np.float32)
    v = v[np.abs(v) <= 448.0]
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_double(float(a)) for a in v], np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_round_trip_and_saturation():
    for b in range(256):
        if (b & 0x7F) == 0x7F:
            continue                                                    # NaN codes
        v = oracle.e4m3_to_double(b)
        assert oracle.e4m3_from_double(v) == b                          # -0.0 keeps its sign
    assert oracle.e4m3_to_double(0x7E) == 448.0 and oracle.e4m3_to_double(0x01) == 2.0 ** -9
    for v in (448.0, 449.0, 480.0, 1e30):
        assert oracle.e4m3_from_double(v) == 0x7E and oracle.e4m3_from_double(-v) == 0xFE


def test_mxfp8_scale_rule_and_error_bound():
    w_ = ms.workload("prefill")
    x = ms.gen_x(w_, T=4)[0]
    xf = ms.f32_from_bf16_bits(x).astype(np.float64)
    for t in range(4):
        codes, scales = oracle.quantize_mxfp8(x[t])
        for b in range(w_.H // 32):
            blk = xf[t, 32 * b:32 * (b + 1)]
            amax = np.abs(blk).max()
            se = (math.frexp(amax)[1] - 1) - 8                          # floor(log2 amax) - 8
            assert scales[b] == se + 127
            X = 2.0 ** se
            deq = np.array([oracle.e4m3_to_double(c) for c in codes[32 * b:32 * (b + 1)]]) * X
            sat = np.abs(blk) > 448 * X
            bound = np.maximum(np.abs(blk) * 2.0 ** -4, X * 2.0 ** -10)
            assert np.all(np.abs(deq - blk)[~sat] <= bound[~sat])
            assert np.all(np.abs(deq[sat]) == 448 * X)


def test_pack_mxfp8_places_quantized_rows():
    w_ = ms.workload("tiny")
    inp = ms.gen_inputs(w_)
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap = w_.T * min(w_.k, w_.P)
    q, src, st = oracle.dispatch_pack_mxfp8(inp["x"], lay["token_slot"], cap)
    assert st == 0
    used = lay["part_offsets"][0, -1]
    for r in (0, 7, used - 1):
        codes, scales = oracle.quantize_mxfp8(inp["x"][0, src[0, r]])
        assert np.array_equal(q[0, r], np.concatenate([codes, scales]))
    _, src_bf16, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap)
    assert np.array_equal(src, src_bf16)
    assert np.all(q[0, used:] == 0)                                      # unused rows untouched


def test_expert_scale_mxfp8_hand_values():
    # two records of H = 32: codes and scale bytes chosen by hand, values worked out
    # from the E4M3 / E8M0 definitions (1.m x 2^(E-7); 2^(byte-127))
    H = 32
    rec = np.zeros((3, H + 1), np.uint8)
    rec[0, :4] = [0x7E, 0x38, 0xB0, 0x01]     # 448, 1.0, -0.5, 2^-9
    rec[0, H] = 127                            # X = 1
    rec[1, :2] = [0x3C, 0xFE]                  # 1.5, -448
    rec[1, H] = 127 + 3                        # X = 8
    rec[2, :] = 0x38
    rec[2, H] = 127
    eo = np.array([0, 1, 2], np.int32)         # expert 0: row 0; expert 1: row 1; row 2 outside
    y = oracle.expert_scale_mxfp8(rec, eo, np.array([1.0, 0.5], np.float32),
                                  y=np.full((3, H), 0x1234, np.uint16))
    got = ms.f32_from_bf16_bits(y).astype(np.float64)
    assert list(got[0, :4]) == [448.0, 1.0, -0.5, 2.0 ** -9] and np.all(got[0, 4:] == 0)
    assert list(got[1, :2]) == [1.5 * 8 * 0.5, -448 * 8 * 0.5] and np.all(got[1, 2:] == 0)
    assert np.all(y[2] == 0x1234)


def test_expert_scale_mxfp8_reduces_to_bf16_expert():
    # a record whose values are all exact in E4M3 dequantizes to those values: the
    # quantized expert must then equal the bf16 expert on the same rows
    rng = np.random.default_rng(3)
    H, R = 64, 40
    mant = rng.integers(8, 16, size=(R, H))                # 1.m in eighths: 3 mantissa bits
    expo = rng.integers(-3, 3, size=(R, H))                # |v| <= 7.5
    v = np.where(rng.random((R, H)) < 0.5, -1.0, 1.0) * mant / 8.0 * 2.0 ** expo
    v[:, ::32] = 14.0 * np.sign(v[:, ::32])                # amax 14 per block: X = 2^-5, 14/X = 448
    bits = ms.bf16_bits_from_f32(v.astype(np.float32))
    rec = np.stack([np.concatenate(oracle.quantize_mxfp8(r)) for r in bits])
    assert np.all(rec[:, H:] == 127 - 5)
    eo = np.array([0, 17, R], np.int32)
    s = np.array([0.25, 3.0], np.float32)
    assert np.array_equal(oracle.expert_scale_mxfp8(rec, eo, s), oracle.expert_scale(bits, eo, s))


# ------------------------------ expert placement and copies (b1g section 6) --

def _check_plan_invariants(load, P, R, plan):
    E = load.size
    Lb, Lp = E // P, E // P + R
    co, cs, se = plan["copy_offsets"], plan["copy_slots"], plan["slot_expert"]
    assert co[0] == 0 and np.all(np.diff(co) >= 1)               # every expert has a slot
    assert co[-1] <= E + P * R
    for e in range(E):
        sl = cs[co[e]:co[e + 1]]
        assert np.all(se[sl] == e)
        assert len(set(sl // Lp)) == sl.size                     # one copy per partition at most
        assert sl[0] % Lp < Lb                                   # the original in a regular slot
        assert np.all(sl[1:] % Lp >= Lb)                         # copies in spare slots
    assert np.sum(se >= 0) == co[-1]
    # loads: the even split of every expert over its copies, summed per partition
    want = np.zeros(P, np.int64)
    for e in range(E):
        n = co[e + 1] - co[e]
        for c, s_ in enumerate(cs[co[e]:co[e + 1]]):
            want[s_ // Lp] += len(range(c, int(load[e]), n))
    assert np.array_equal(plan["part_load"], want)
    assert plan["part_load"].sum() == load.sum()


def test_placement_hand_example():
    g = _golden("placement_hand.json")
    load = np.array(g["load"], np.int64)
    plan = oracle.plan_placement(load, g["P"], g["R"])
    for key in ("copy_offsets", "copy_slots", "slot_expert", "part_load"):
        assert plan[key].tolist() == g[key], key
    _check_plan_invariants(load, g["P"], g["R"], plan)


@pytest.mark.parametrize("E,P,R,seed", [(16, 4, 0, 1), (16, 4, 2, 2), (64, 8, 4, 3),
                                        (384, 8, 4, 4), (8, 8, 3, 5), (64, 64, 1, 6)])
def test_placement_invariants_and_gain(E, P, R, seed):
    rng = np.random.default_rng(seed)
    p = (np.arange(E) + 1.0) ** -1.2
    load = rng.multinomial(E * 40, p / p.sum()).astype(np.int64)
    rng.shuffle(load)
    plan = oracle.plan_placement(load, P, R)
    _check_plan_invariants(load, P, R, plan)
    # contiguous placement (expert e on partition e // (E/P)) as the baseline
    base = np.bincount(np.arange(E) // (E // P), weights=load, minlength=P)
    only = oracle.plan_placement(load, P, 0)
    assert only["copy_offsets"][-1] == E                          # R = 0: no copies
    assert plan["part_load"].max() <= only["part_load"].max()     # copies never raise the max
    if E > P:
        assert only["part_load"].max() <= base.max()              # greedy beats contiguous here
    else:
        # one expert per partition: placement cannot help, only copies can
        assert only["part_load"].max() == load.max()
        if R > 0:
            assert plan["part_load"].max() < load.max()


def test_map_replicas_identity_and_skips():
    rng = np.random.default_rng(11)
    E = 16
    ids = rng.integers(-1, E + 2, size=(2, 50, 3)).astype(np.int32)
    co, cs = np.arange(E + 1, dtype=np.int32), np.arange(E, dtype=np.int32)
    phys = oracle.map_replicas(ids, E, co, cs, E)
    assert np.array_equal(phys[(ids >= 0) & (ids < E)], ids[(ids >= 0) & (ids < E)])
    assert np.all(phys[ids < 0] == -1) and np.all(phys[ids >= E] == E)


def test_map_replicas_round_robin_split():
    # one expert per partition and skewed popularity, so the plan copies hot experts
    rng = np.random.default_rng(12)
    E, P, R = 8, 8, 2
    pop = (np.arange(E) + 1.0) ** -1.5
    ids = np.stack([np.stack([rng.choice(E, size=4, replace=False, p=pop / pop.sum())
                              for _ in range(200)]) for _ in range(3)]).astype(np.int32)
    load = np.bincount(ids[0].ravel(), minlength=E).astype(np.int64)
    plan = oracle.plan_placement(load, P, R)
    co, cs = plan["copy_offsets"], plan["copy_slots"]
    assert co[-1] > E                                             # copies were made
    phys = oracle.map_replicas(ids, E, co, cs, plan["E_phys"])
    assert np.array_equal(plan["slot_expert"][phys], ids)         # a copy of the right expert
    for s in range(3):
        flat_ids, flat_ph = ids[s].ravel(), phys[s].ravel()       # (t, j) order
        for e in range(E):
            got = flat_ph[flat_ids == e]
            n = co[e + 1] - co[e]
            want = cs[co[e] + np.arange(got.size) % n]            # r-th pair -> copy r mod n
            assert np.array_equal(got, want)
    # on the batch the plan was made from, the partition loads are the plan's
    lay = oracle.dispatch_layout(phys[:1], plan["E_phys"], P)
    pairs_per_part = lay["expert_counts"][0].reshape(P, -1).sum(axis=1)
    assert np.array_equal(pairs_per_part, plan["part_load"])


def test_placement_rejects_a_copy_that_ties_the_busiest():
    # e0 (6) on p0, e1 (3) on p1; copying e0 to p1 would give p1 3 + 3 = 6, equal to the
    # busiest partition's 6: that is a new busiest partition, so no copy is kept
    plan = oracle.plan_placement(np.array([6, 3], np.int64), 2, 1)
    assert plan["copy_offsets"].tolist() == [0, 1, 2] and plan["part_load"].tolist() == [6, 3]
    # with 7 the copy brings p1 to 3 + 3 = 6 < 7 and is kept; p0 keeps the larger share
    plan = oracle.plan_placement(np.array([7, 3], np.int64), 2, 1)
    assert plan["copy_offsets"].tolist() == [0, 2, 3] and plan["part_load"].tolist() == [4, 6]


def test_placed_path_output_equals_unplaced():
    # copies of an expert compute what the expert computes, so moving pairs between
    # copies (and experts between partitions) leaves the combined output unchanged
    w_ = ms.workload("tiny", E=32, P=32, k=4, zipf_s=1.2, T=600)
    inp = ms.gen_inputs(w_)
    ids, wts = oracle.route_topk(inp["logits"], w_.k)
    plan = oracle.plan_placement(np.bincount(ids.ravel(), minlength=w_.E).astype(np.int64), w_.P, 2)
    assert plan["copy_offsets"][-1] > w_.E
    phys = oracle.map_replicas(ids, w_.E, plan["copy_offsets"], plan["copy_slots"], plan["E_phys"])
    lay = oracle.dispatch_layout(phys, plan["E_phys"], w_.P)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], w_.T * min(w_.k, w_.P))
    per = oracle.permute_to_experts(send, lay["token_slot"], phys, plan["E_phys"])
    se = plan["slot_expert"]
    y = oracle.expert_scale(per["recv"], per["expert_offsets"],
                            np.where(se >= 0, inp["scales"][np.maximum(se, 0)], 0).astype(np.float32))
    ref = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, inp["scales"])
    assert np.array_equal(oracle.combine(y, per["pair_row"], wts), ref["out"])
    # and the busiest partition carries less than under contiguous blocks
    cont = np.bincount(ids.ravel(), minlength=w_.E).reshape(w_.P, -1).sum(axis=1)
    placed = lay["expert_counts"][0].reshape(w_.P, -1).sum(axis=1)
    assert placed.max() < cont.max()


# ------------------------------------------- routed payload (a2a 6.1, 7.1) --

def _routed_case(name, **over):
    w_ = ms.workload(name, **over)
    inp = ms.gen_inputs(w_)
    ids, wts = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap = w_.T * min(w_.k, w_.P) + 3                       # three rows no slot names
    return w_, inp, ids, wts, lay, cap


def test_routed_pack_carries_the_tokens_routing():
    w_, inp, ids, wts, lay, cap = _routed_case("tiny", S=2, T=90)
    send, src, sid, sw, st = oracle.dispatch_pack_routed(inp["x"], ids, wts, lay["token_slot"], cap)
    ref_send, ref_src, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap)
    assert st == 0 and np.array_equal(send, ref_send) and np.array_equal(src, ref_src)
    for s in range(w_.S):
        used = src[s] >= 0
        assert np.array_equal(sid[s][used], ids[s][src[s][used]])
        assert np.array_equal(sw[s][used], wts[s][src[s][used]].astype(np.float32))
        assert np.all(sid[s][~used] == -1) and np.all(sw[s][~used] == 0)
        assert (~used).sum() >= 3


@pytest.mark.parametrize("name,over,recv_part", [("tiny", {}, -1), ("tiny", {"S": 3, "T": 70}, 1),
                                                 ("decode", {}, -1), ("decode", {}, 6)])
def test_routed_stage1_equals_permuted_stage1(name, over, recv_part):
    # two formulations of the per-partition pre-add: over rows in arrival order with
    # their ids (routed), and over the expert-sorted pair rows (permute + stand-in expert)
    w_, inp, ids, wts, lay, cap = _routed_case(name, **over)
    send, _, sid, sw, _ = oracle.dispatch_pack_routed(inp["x"], ids, wts, lay["token_slot"], cap)
    fill = np.full_like(send, 0x1357)
    got, st = oracle.routed_expert_stage1(send, sid, sw, lay["part_offsets"], w_.E, recv_part,
                                          inp["scales"], ret=fill.copy())
    per = oracle.permute_to_experts(send, lay["token_slot"], ids, w_.E, recv_part=recv_part)
    y = oracle.expert_scale(per["recv"], per["expert_offsets"], inp["scales"])
    want, st2 = oracle.combine_stage1(y, per["pair_row"], wts, ids, lay["token_slot"], w_.E, cap,
                                      recv_part=recv_part, ret=fill.copy())
    assert st == st2 == 0
    assert np.array_equal(got, want)


def test_routed_round_trip_is_the_combine():
    w_, inp, ids, wts, lay, cap = _routed_case("decode")
    send, _, sid, sw, _ = oracle.dispatch_pack_routed(inp["x"], ids, wts, lay["token_slot"], cap)
    ret, _ = oracle.routed_expert_stage1(send, sid, sw, lay["part_offsets"], w_.E)
    out, st = oracle.combine_stage2(ret, lay["token_slot"])
    assert st == 0
    # identity expert: the per-partition weights add up to 1, so out ~ x
    x = ms.f32_from_bf16_bits(inp["x"]).astype(np.float64)
    got = ms.f32_from_bf16_bits(out).astype(np.float64)
    assert np.all(np.abs(got - x) <= 2.0 ** -6 * np.maximum(np.abs(x), 1e-3))


def test_routed_stage1_skips_empty_and_flags_bad_ids():
    w_, inp, ids, wts, lay, cap = _routed_case("tiny", T=40)
    send, _, sid, sw, _ = oracle.dispatch_pack_routed(inp["x"], ids, wts, lay["token_slot"], cap)
    sid = sid.copy()
    r0 = int(lay["part_offsets"][0, 2])                    # first row of partition 2
    sid[0, r0, 0] = w_.E + 4
    fill = np.full_like(send, 0x2468)
    ret, st = oracle.routed_expert_stage1(send, sid, sw, lay["part_offsets"], w_.E, ret=fill.copy())
    assert st == oracle.BIT_BAD_ID
    used = int(lay["part_offsets"][0, -1])
    assert np.all(ret[0, used:] == 0x2468)                 # empty rows are not written


# ------------------------------------------------- NVFP4 rows (a2a 7.2) --

def test_e2m1_table_ties_and_saturation():
    # E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit -> 0, 0.5, 1, 1.5, 2, 3, 4, 6
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [oracle.e2m1_to_double(c) for c in range(8)] == mags
    assert [oracle.e2m1_to_double(c + 8) for c in range(8)] == [-m for m in mags]
    for c in range(16):
        assert oracle.e2m1_from_double(oracle.e2m1_to_double(c)) == c     # -0 keeps its sign
    # midpoints go to the code with mantissa bit 0
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, want in ties.items():
        assert oracle.e2m1_to_double(oracle.e2m1_from_double(v)) == want
        assert oracle.e2m1_to_double(oracle.e2m1_from_double(-v)) == -want
    for v in (6.0, 6.5, 7.0, 1e30):
        assert oracle.e2m1_from_double(v) == 7 and oracle.e2m1_from_double(-v) == 15
    assert oracle.e2m1_from_double(0.2) == 0 and oracle.e2m1_from_double(-0.2) == 8


def test_nvfp4_row_size_and_hand_block():
    g = _golden("quantized_row_bytes.json")
    H = g["hidden"]
    codes, scales = oracle.quantize_nvfp4(ms.gen_x(ms.workload("prefill"), T=1)[0, 0])
    assert codes.nbytes + scales.nbytes == g["nvfp4_bytes"]                # 1 B scale per 16
    ts = np.zeros((1, 1, 1), np.int32)
    q, _, _ = oracle.dispatch_pack_nvfp4(ms.gen_x(ms.workload("prefill"), T=1), ts, 1)
    assert q.shape == (1, 1, g["nvfp4_bytes"])
    # a block with max |v| = 6: s = e4m3(6/6) = 1.0 (byte 0x38), codes are e2m1(v)
    v = np.zeros(16, np.float32)
    v[:8] = [6.0, 3.0, -1.5, 0.25, 0.75, -5.0, 0.5, 2.5]
    c, s = oracle.quantize_nvfp4(ms.bf16_bits_from_f32(v))
    assert s.tolist() == [0x38]
    nib = [(c[i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
    assert [oracle.e2m1_to_double(n) for n in nib[:8]] == [6.0, 3.0, -1.5, 0.0, 1.0, -4.0, 0.5, 2.0]
    assert nib[8:] == [0] * 8
    # max |v| = 12: s = 2 (byte 0x40), 9 -> 4.5 -> 4 (tie at 5? no: 4.5 is between 4 and 6 -> 4)
    v = np.zeros(16, np.float32)
    v[:3] = [12.0, 9.0, -0.5]
    c, s = oracle.quantize_nvfp4(ms.bf16_bits_from_f32(v))
    assert s.tolist() == [0x40]
    nib = [(c[i // 2] >> (4 * (i % 2))) & 0xF for i in range(3)]
    assert [oracle.e2m1_to_double(n) * 2.0 for n in nib] == [12.0, 8.0, -0.0]
    # an all-zero block: scale byte 0 and zero codes
    c, s = oracle.quantize_nvfp4(np.zeros(16, np.uint16))
    assert s.tolist() == [0] and c.tolist() == [0] * 8


@pytest.mark.parametrize("g", [1.0, 2.0 ** -12, 0.37])
def test_nvfp4_error_bound(g):
    rng = np.random.default_rng(21)
    x = ms.bf16_bits_from_f32((rng.standard_normal((64, 256)) * np.exp(rng.uniform(-6, 6, (64, 1))))
                              .astype(np.float32))
    flushed = 0
    for t in range(64):
        codes, scales = oracle.quantize_nvfp4(x[t], g)
        vals = ms.f32_from_bf16_bits(x[t]).astype(np.float64)
        for b in range(16):
            sg = oracle.e4m3_to_double(int(scales[b])) * g
            blk = vals[16 * b:16 * (b + 1)]
            nib = [(codes[8 * b + i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
            deq = np.array([oracle.e2m1_to_double(n) for n in nib]) * sg
            if sg == 0:
                # the block scale rounds to zero only below half the smallest E4M3 value
                assert np.abs(blk).max() / (6 * g) <= 2.0 ** -10 and np.all(deq == 0)
                flushed += 1
                continue
            q = np.abs(blk) / sg
            # half the E2M1 spacing (0.25 below 2, q/4 above), plus what saturation at 6 cuts
            bound = sg * (np.maximum(0.25, q / 4) + np.maximum(0.0, q - 6)) * (1 + 1e-6)
            assert np.all(np.abs(deq - blk) <= bound)
    if g == 1.0:
        assert flushed > 0          # the tensor scale is what keeps small blocks alive
    if g == 2.0 ** -12:
        assert flushed == 0


def test_expert_scale_nvfp4_reduces_to_bf16_expert():
    rng = np.random.default_rng(4)
    H, R = 64, 30
    mags = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0])
    v = rng.choice(mags, size=(R, H)) * np.where(rng.random((R, H)) < 0.5, -1, 1)
    v[:, ::16] = 6.0                                       # amax 6 per block: s = 1 exactly
    bits = ms.bf16_bits_from_f32(v.astype(np.float32))
    rec = np.stack([np.concatenate(oracle.quantize_nvfp4(r)) for r in bits])
    assert np.all(rec[:, H // 2:] == 0x38)
    eo = np.array([0, 11, R], np.int32)
    s = np.array([0.75, 2.5], np.float32)
    assert np.array_equal(oracle.expert_scale_nvfp4(rec, eo, s), oracle.expert_scale(bits, eo, s))
    # the same values at a tensor scale of 2^-3: scales step up by 3 binades, output unchanged
    rec3 = np.stack([np.concatenate(oracle.quantize_nvfp4(r, 0.125)) for r in bits])
    assert np.all(rec3[:, H // 2:] == 0x38 + (3 << 3))
    assert np.array_equal(oracle.expert_scale_nvfp4(rec3, eo, s, g=0.125), oracle.expert_scale(bits, eo, s))
