"""Pins of the CPU oracle against facts outside it.

Each check below compares the oracle with something it does not contain:
a hand-worked fixture, a library routine (a stable sort, a softmax, a
dense matmul of the dequantised bank -- the page's eager reference), a
closed form or an invariant.  A dropped term, a wrong sign or index or a
transposed operand anywhere in the oracle fails at least one of them.
"""
import os

import numpy as np
import pytest
import scipy.special

import oracle
from bit_moe_expert_router_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TINY = synth.WORKLOADS["tiny"]


def _lut():
    """Byte -> (low code, high code) table built from the oracle's unpack (pinned below)."""
    return np.array([[oracle.unpack(b, 0), oracle.unpack(b, 1)] for b in range(256)], dtype=np.int64)


def _dequant(codes, scales, g):
    """Dense fp64 weights: code * scale of its (row, group)."""
    return codes.astype(np.float64) * np.repeat(scales.astype(np.float64), g, axis=-1)


@pytest.fixture(scope="module")
def tiny():
    bank, c13, c2 = synth.make_bank(TINY, with_codes=True)
    return bank, c13, c2, synth.make_tokens(TINY)


# ----------------------------------------------------------------- storage format

def test_unpack_matches_hand_worked_bytes():
    rows = []
    with open(os.path.join(GOLDEN, "int4_nibbles.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                b, lo, hi = line.split()
                rows.append((int(b, 16), int(lo), int(hi)))
    assert len(rows) >= 10
    for b, lo, hi in rows:
        assert oracle.unpack(b, 0) == lo and oracle.unpack(b, 1) == hi, hex(b)


def test_every_byte_round_trips_through_codes():
    lut = _lut()
    assert lut.min() == -8 and lut.max() == 7
    rebuilt = (lut[:, 0] & 0xF) | ((lut[:, 1] & 0xF) << 4)
    assert np.array_equal(rebuilt, np.arange(256))


def test_generator_bank_bytes_hold_its_codes(tiny):
    bank, c13, c2, _ = tiny
    lut = _lut()
    for packed, codes in ((bank.w13, c13), (bank.w2, c2)):
        unpacked = lut[packed].reshape(*packed.shape[:-1], -1)  # [..., K/2, 2] -> [..., K]
        assert np.array_equal(unpacked, codes)


# ----------------------------------------------------------------- route

def _softmax_topk_renorm(logits, k):
    """The recipe's order: full softmax, then top-k of the probabilities, then renormalise."""
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    ids = np.argsort(-p, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(p, ids, axis=1)
    return ids, sel / sel.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("name,k", [("tiny", 2), ("decode_t4", 10), ("large_bank_t2048", 8)])
def test_route_equals_softmax_topk_renormalise(name, k):
    w = synth.WORKLOADS[name].with_tokens(64)
    logits = synth.make_tokens(w).logits
    ids, wt = oracle.route(logits, k)
    ids_ref, w_ref = _softmax_topk_renorm(logits, k)
    assert np.array_equal(ids, ids_ref)
    assert np.max(np.abs(wt - w_ref)) < 1e-12
    assert np.max(np.abs(wt.sum(axis=1) - 1.0)) < 1e-12
    # descending logits along j
    sel = np.take_along_axis(logits, ids, axis=1)
    assert np.all(np.diff(sel, axis=1) <= 0)


def test_route_ties_go_to_lower_index():
    l = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.0, -0.0, 0.0]], dtype=np.float32)
    ids, w = oracle.route(l, 8)
    assert ids[0].tolist() == [1, 2, 4, 3, 0, 5, 6, 7]
    ids3, w3 = oracle.route(l, 3)
    assert ids3[0].tolist() == [1, 2, 4]
    assert np.allclose(w3, 1.0 / 3.0, rtol=0, atol=1e-15)
    ids6, _ = oracle.route(l, 6)
    assert ids6[0].tolist() == [1, 2, 4, 3, 0, 5]
    # the same order as a stable sort of the negated logits (a library routine)
    assert ids[0].tolist() == np.argsort(-l[0], kind="stable").tolist()


def test_route_k1_and_k_equals_E():
    logits = synth.make_tokens(TINY).logits
    ids1, w1 = oracle.route(logits, 1)
    assert np.array_equal(ids1[:, 0], np.argmax(logits, axis=1))
    assert np.all(w1 == 1.0)
    idsE, wE = oracle.route(logits, TINY.E)
    assert np.array_equal(idsE, np.argsort(-logits, axis=1, kind="stable"))
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.max(np.abs(wE - np.take_along_axis(full, idsE, axis=1))) < 1e-12


def test_route_orders_nan_logits_last():
    """NaN ranks below every number (-inf included), NaNs by index: numpy's stable lexsort on (is NaN, -value)."""
    rng = np.random.default_rng(11)
    l = rng.standard_normal((40, 24)).astype(np.float32)
    l[rng.random(l.shape) < 0.25] = np.nan
    l[0, :] = np.nan                       # all NaN: the lowest indices
    l[1, :5] = -np.inf
    l[1, 5:] = np.nan                      # -inf before every NaN
    l[2, 3] = np.inf
    for k in (1, 5, 24):
        ids, _ = oracle.route(l, k)
        ref = np.stack([np.lexsort((np.where(np.isnan(r), 0.0, -r.astype(np.float64)), np.isnan(r)))[:k] for r in l])
        assert np.array_equal(ids, ref), k
        assert all(len(set(row)) == k for row in ids.tolist())
    assert oracle.route(l, 3)[0][0].tolist() == [0, 1, 2]
    assert oracle.route(l, 6)[0][1].tolist() == [0, 1, 2, 3, 4, 5]


def test_route_rejects_bad_k():
    with pytest.raises(ValueError):
        oracle.route(np.zeros((2, 4), np.float32), 5)


# ----------------------------------------------------------------- permute

@pytest.mark.parametrize("name", ["tiny", "prefill_t8192"])
def test_permute_equals_stable_sort(name):
    w = synth.WORKLOADS[name].with_tokens(min(synth.WORKLOADS[name].T, 512))
    ids, _ = oracle.route(synth.make_tokens(w).logits, w.top_k)
    counts, offsets, perm, inv = oracle.permute(ids, w.E)
    flat = ids.ravel()
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(counts, np.bincount(flat, minlength=w.E))
    assert offsets[0] == 0 and offsets[-1] == flat.size
    assert np.array_equal(offsets[1:], np.cumsum(counts))
    assert np.array_equal(perm[inv], np.arange(flat.size))
    assert np.array_equal(np.bincount(perm // w.top_k, minlength=w.T), np.full(w.T, w.top_k))
    for e in range(w.E):  # stable: increasing within each expert's run
        run = perm[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(run) > 0)
        assert np.all(flat[run] == e)


def test_permute_empty_and_single_expert():
    counts, offsets, perm, inv = oracle.permute(np.zeros((0, 2), np.int32), 4)
    assert counts.tolist() == [0, 0, 0, 0] and offsets.tolist() == [0] * 5 and perm.size == 0
    ids = np.full((5, 1), 3, np.int32)
    counts, offsets, perm, inv = oracle.permute(ids, 4)
    assert counts.tolist() == [0, 0, 0, 5] and perm.tolist() == [0, 1, 2, 3, 4]


# ----------------------------------------------------------------- projections

def test_partials_equal_integer_matmul(tiny):
    bank, c13, c2, tok = tiny
    g = TINY.group
    for t, e in [(0, 0), (5, 3), (15, 7)]:
        P = oracle.partials(tok.x_q[t], bank.w13[e], g)
        a = tok.x_q[t].astype(np.int64).reshape(-1, g)
        ref = np.einsum("qk,nqk->nq", a, c13[e].astype(np.int64).reshape(c13.shape[1], -1, g))
        assert np.array_equal(P, ref)


def test_partials_extremes_do_not_overflow():
    g, K = 128, 4096
    a = np.full(K, -127, np.int8)
    W = np.full((3, K // 2), 0x88, np.uint8)  # every code -8
    P = oracle.partials(a, W, g)
    assert np.all(P == g * 127 * 8)


def test_one_hot_activation_selects_a_column(tiny):
    bank, c13, _, _ = tiny
    H, I, g = TINY.H, TINY.I, TINY.group
    e, c = 2, 77
    x = np.zeros(H, np.int8)
    x[c] = 1
    _, G, _ = oracle.hidden(x, 1.0, bank.w13[e], bank.s13[e], g)
    expect = c13[e][:, c].astype(np.float64) * bank.s13[e][:, c // g].astype(np.float64)
    assert np.array_equal(G, expect)


def test_hidden_equals_dequantised_matmul(tiny):
    """The page's eager reference: dequantise the packed bank, then a plain matmul."""
    bank, c13, _, tok = tiny
    I, g = TINY.I, TINY.group
    for t, e in [(0, 1), (7, 4), (15, 6)]:
        P1, G, h = oracle.hidden(tok.x_q[t], tok.x_scale[t], bank.w13[e], bank.s13[e], g)
        W = _dequant(c13[e], bank.s13[e], g)
        G_ref = W @ (tok.x_q[t].astype(np.float64) * np.float64(tok.x_scale[t]))
        scale = np.max(np.abs(G_ref))
        assert np.max(np.abs(G - G_ref)) <= 1e-12 * scale
        h_ref = G_ref[:I] * scipy.special.expit(G_ref[:I]) * G_ref[I:]
        assert np.max(np.abs(h - h_ref)) <= 1e-12 * np.max(np.abs(h_ref))


def test_silu_matches_library():
    z = np.concatenate([np.linspace(-30, 30, 601), [0.0, 1e-300, -1e-300, 700.0, -700.0]])
    ref = z * scipy.special.expit(z)
    got = np.array([oracle.silu(v) for v in z])
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-300)


def test_requant_rounds_half_to_even():
    # amax 127 gives s_h = 1 exactly, so h / s_h is h itself.
    h = np.array([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 63.5, 64.5, -126.5, 0.0])
    hq, sh = oracle.requant(h)
    assert sh == 1.0
    assert hq.tolist() == [127, 0, 2, 2, 0, -2, -2, 64, 64, -126, 0]
    hq0, sh0 = oracle.requant(np.zeros(8))
    assert sh0 == 0.0 and not hq0.any()


def test_requant_code_range_and_scale(tiny):
    _, _, _, tok = tiny
    rng = np.random.default_rng(3)
    for _ in range(20):
        h = rng.standard_normal(128) * rng.uniform(1e-6, 1e3)
        hq, sh = oracle.requant(h)
        assert np.max(np.abs(hq.astype(int))) == 127
        assert sh == np.float32(np.max(np.abs(h.astype(np.float32)))) / np.float32(127)
        # each code is within half a step of the value it encodes
        assert np.all(np.abs(hq * np.float64(sh) - h) <= 0.5 * sh * (1 + 1e-6) + 1e-30)


def test_down_equals_dequantised_matmul(tiny):
    bank, _, c2, tok = tiny
    g = TINY.group
    rng = np.random.default_rng(1)
    for e in [0, 3, 7]:
        hq = rng.integers(-127, 128, TINY.I).astype(np.int8)
        sh = 0.0123
        P2, y = oracle.down(hq, sh, bank.w2[e], bank.s2[e], g)
        y_ref = _dequant(c2[e], bank.s2[e], g) @ (hq.astype(np.float64) * np.float64(np.float32(sh)))
        assert np.max(np.abs(y - y_ref)) <= 1e-12 * np.max(np.abs(y_ref))
        ref_P = np.einsum("qk,nqk->nq", hq.astype(np.int64).reshape(-1, g),
                          c2[e].astype(np.int64).reshape(c2.shape[1], -1, g))
        assert np.array_equal(P2, ref_P)


def test_identity_down_projection_returns_dequantised_h():
    I = H = 64
    g = 64
    codes = np.eye(H, I, dtype=np.int64)
    w2 = ((codes[:, 0::2] & 0xF) | ((codes[:, 1::2] & 0xF) << 4)).astype(np.uint8)
    s2 = np.ones((H, I // g), np.float32)
    hq = np.arange(-32, 32, dtype=np.int8)
    _, y = oracle.down(hq, 0.5, w2, s2, g)
    assert np.array_equal(y, hq.astype(np.float64) * 0.5)


# ----------------------------------------------------------------- whole layer

def _brute_force_layer(w, tok, bank, c13, c2):
    """Dense numpy restatement: library softmax/top-k, dequantised matmuls, library SiLU and RNE."""
    ids, wt = _softmax_topk_renorm(tok.logits, w.top_k)
    x = tok.x_q.astype(np.float64) * tok.x_scale.astype(np.float64)[:, None]
    out = np.zeros((w.T, w.H))
    for t in range(w.T):
        slots = list(ids[t]) + list(range(w.E, w.E + w.S))
        weights = list(wt[t]) + [1.0] * w.S
        for slot, wj in zip(slots, weights):
            G = _dequant(c13[slot], bank.s13[slot], w.group) @ x[t]
            h = (G[:w.I] * scipy.special.expit(G[:w.I]) * G[w.I:]).astype(np.float32)
            sh = np.float32(np.max(np.abs(h))) / np.float32(127)
            hq = np.clip(np.rint(h / sh), -127, 127) if sh > 0 else np.zeros_like(h)
            y = _dequant(c2[slot], bank.s2[slot], w.group) @ (hq.astype(np.float64) * np.float64(sh))
            out[t] += wj * y
    return out


def test_layer_equals_brute_force(tiny):
    bank, c13, c2, tok = tiny
    out = oracle.forward_workload(TINY, tok, bank)
    ref = _brute_force_layer(TINY, tok, bank, c13, c2)
    assert np.max(np.abs(out - ref)) <= 1e-9 * np.sqrt(np.mean(ref ** 2))


def test_layer_with_shared_expert_equals_brute_force():
    w = synth.Workload("t", T=6, H=256, I=128, E=6, S=1, top_k=3, group=128, bias="zipf", zipf_s=1.0)
    bank, c13, c2 = synth.make_bank(w, with_codes=True)
    tok = synth.make_tokens(w)
    out = oracle.forward_workload(w, tok, bank)
    ref = _brute_force_layer(w, tok, bank, c13, c2)
    assert np.max(np.abs(out - ref)) <= 1e-9 * np.sqrt(np.mean(ref ** 2))
    # the shared slot adds its own output with weight 1
    d0 = oracle.dims(w.T, w.H, w.I, w.E, 0, w.top_k, w.group)
    routed = oracle.forward_tokens(d0, tok.x_q, tok.x_scale, tok.logits, bank.w13, bank.s13, bank.w2, bank.s2)
    d = oracle.dims(w.T, w.H, w.I, w.E, 1, w.top_k, w.group)
    for t in range(w.T):
        _, _, y = oracle.pair_output(d, tok.x_q, tok.x_scale, bank.w13, bank.s13, bank.w2, bank.s2, t, w.E)
        assert np.max(np.abs(out[t] - routed[t] - y)) <= 1e-12 * np.max(np.abs(out[t]))


def test_dense_case_E1_k1(tiny):
    """One expert, top-1, no shared expert: a single dense W4A8 MLP per token."""
    bank, c13, c2, tok = tiny
    w = synth.Workload("dense", T=TINY.T, H=TINY.H, I=TINY.I, E=1, S=0, top_k=1, group=TINY.group)
    sub = synth.Bank(bank.w13[:1], bank.s13[:1], bank.w2[:1], bank.s2[:1], bank.twobit[:1])
    tok1 = synth.Tokens(tok.x_q, tok.x_scale, tok.logits[:, :1].copy())
    out = oracle.forward_workload(w, tok1, sub)
    ref = _brute_force_layer(w, tok1, sub, c13[:1], c2[:1])
    assert np.max(np.abs(out - ref)) <= 1e-9 * np.sqrt(np.mean(ref ** 2))


def test_zero_weight_expert_contributes_zero(tiny):
    bank, _, _, tok = tiny
    z13, z2 = bank.w13.copy(), bank.w2.copy()
    zs13, zs2 = bank.s13.copy(), bank.s2.copy()
    z13[3] = 0
    z2[3] = 0
    zs13[3] = 0
    zs2[3] = 0
    d = oracle.dims(TINY.T, TINY.H, TINY.I, TINY.E, 0, TINY.top_k, TINY.group)
    hq, sh, y = oracle.pair_output(d, tok.x_q, tok.x_scale, z13, zs13, z2, zs2, 0, 3)
    assert sh == 0.0 and not hq.any() and not y.any()
    # only the other expert of a token routed to slot 3 remains
    ids, wt = oracle.route(tok.logits, TINY.top_k)
    out = oracle.forward_tokens(d, tok.x_q, tok.x_scale, tok.logits, z13, zs13, z2, zs2)
    for t in np.nonzero((ids == 3).any(axis=1))[0]:
        j = int(np.nonzero(ids[t] != 3)[0][0])
        _, _, y_other = oracle.pair_output(d, tok.x_q, tok.x_scale, z13, zs13, z2, zs2, int(t), int(ids[t, j]))
        assert np.array_equal(out[t], wt[t, j] * y_other + 0.0) or \
            np.max(np.abs(out[t] - wt[t, j] * y_other)) <= 1e-15 * np.max(np.abs(y_other))


def test_identical_experts_give_that_expert(tiny):
    bank, _, _, tok = tiny
    rep = synth.Bank(np.repeat(bank.w13[:1], TINY.E, 0), np.repeat(bank.s13[:1], TINY.E, 0),
                     np.repeat(bank.w2[:1], TINY.E, 0), np.repeat(bank.s2[:1], TINY.E, 0), bank.twobit)
    out = oracle.forward_workload(TINY, tok, rep)
    d = oracle.dims(TINY.T, TINY.H, TINY.I, TINY.E, 0, TINY.top_k, TINY.group)
    for t in range(TINY.T):
        _, _, y = oracle.pair_output(d, tok.x_q, tok.x_scale, rep.w13, rep.s13, rep.w2, rep.s2, t, 0)
        assert np.max(np.abs(out[t] - y)) <= 1e-12 * np.max(np.abs(y))


def test_token_subset_matches_full_run(tiny):
    bank, _, _, tok = tiny
    full = oracle.forward_workload(TINY, tok, bank)
    sel = np.array([13, 2, 2, 0])
    part = oracle.forward_workload(TINY, tok, bank, sel)
    assert np.array_equal(part, full[sel])


# ----------------------------------------------------------------- generator recipe

def test_generator_activation_codes():
    w = synth.WORKLOADS["decode_verify_t12"]
    tok = synth.make_tokens(w)
    xb = synth.bf16_activations(w)
    assert np.all(np.abs(tok.x_q.astype(int)).max(axis=1) == 127)
    amax = np.abs(xb).max(axis=1)
    assert np.array_equal(tok.x_scale, (amax / np.float32(127)).astype(np.float32))
    # values are bf16: the low 16 bits of the fp32 pattern are zero
    assert not (xb.view(np.uint32) & 0xFFFF).any()
    assert np.all(np.abs(tok.x_q * tok.x_scale[:, None].astype(np.float64) - xb) <= 0.5 * tok.x_scale[:, None] * 1.0001)


def test_generator_weight_code_ranges():
    w = synth.WORKLOADS["large_bank_t2048"]
    small = synth.Workload("lb", T=4, H=256, I=128, E=w.E, S=1, top_k=8, group=128, twobit_frac=0.25)
    bank, c13, c2 = synth.make_bank(small, with_codes=True)
    assert bank.twobit.sum() == 72 and not bank.twobit[small.E]
    for e in range(small.slots):
        lo, hi = (-2, 1) if bank.twobit[e] else (-8, 7)
        assert c13[e].min() >= lo and c13[e].max() <= hi and c2[e].min() >= lo and c2[e].max() <= hi


def test_verify_batch_expert_overlap():
    w0 = synth.WORKLOADS["decode_verify_t12"]
    vals = []
    for seed in range(1, 60):
        w = synth.Workload(**{**w0.__dict__, "seed": seed})
        ids, _ = oracle.route(synth.make_tokens(w).logits, w.top_k)
        for r in range(w.requests):
            for a in range(3):
                for b in range(a + 1, 3):
                    vals.append(len(set(ids[3 * r + a]) & set(ids[3 * r + b])) / w.top_k)
    assert abs(np.mean(vals) - 0.60) < 0.03


def test_zipf_bias_skews_expert_load():
    w = synth.WORKLOADS["prefill_t8192"].with_tokens(1024)
    ids, _ = oracle.route(synth.make_tokens(w).logits, w.top_k)
    counts = np.sort(np.bincount(ids.ravel(), minlength=w.E))[::-1]
    assert counts[0] > 0.5 * w.T and counts[w.E // 2] == 0


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of fp32 values that are exact in bf16 (checked)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def test_s0_quantisation_golden_rows():
    """Hand-worked rows (scales powers of two, half-way cases): exact codes and scales."""
    rows = []
    for line in open(os.path.join(GOLDEN, "s0_quant_bf16.txt")):
        line = line.split("#")[0].split()
        if line:
            rows.append((line[0], [float(v) for v in line[1:]]))
    xs = [v for k, v in rows if k == "x"]
    ss = [v[0] for k, v in rows if k == "s"]
    qs = [v for k, v in rows if k == "q"]
    assert len(xs) == len(ss) == len(qs) == 5
    x_q, x_scale = oracle.quantize_bf16(_bf16_bits(np.array(xs, np.float32)))
    assert np.array_equal(x_scale, np.array(ss, np.float32))
    assert np.array_equal(x_q, np.array(qs, np.int8))


def test_s0_quantisation_matches_the_generators_own_quantiser():
    """Two independent implementations of the same recipe agree bit for bit."""
    for name in ("tiny", "decode_t4", "decode_verify_t12", "large_bank_t2048"):
        w = synth.WORKLOADS[name].with_tokens(min(synth.WORKLOADS[name].T, 64))
        tok = synth.make_tokens(w)
        x_q, x_scale = oracle.quantize_bf16(_bf16_bits(synth.bf16_activations(w)))
        assert np.array_equal(x_scale, tok.x_scale), name
        assert np.array_equal(x_q, tok.x_q), name


def test_s0_quantisation_invariants():
    rng = np.random.default_rng(11)
    T, H = 40, 256
    x = (rng.standard_normal((T, H)) * np.exp(rng.uniform(-20, 20, size=(T, 1)))).astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)  # truncate to bf16
    x[3] = 0.0
    x[4] = -0.0
    x[5, :] = 0.0
    x[5, 17] = -3.0
    x_q, s = oracle.quantize_bf16(_bf16_bits(x))
    assert s[3] == 0 and s[4] == 0 and not x_q[3].any() and not x_q[4].any()
    live = s > 0
    assert np.all(np.abs(x_q.astype(int)) <= 127)
    assert np.all(np.abs(x_q[live].astype(int)).max(axis=1) == 127)
    assert x_q[5, 17] == -127 and np.count_nonzero(x_q[5]) == 1
    # each code is the nearest integer to x / s (within fp32 rounding of the division)
    err = np.abs(x_q[live].astype(np.float64) - x[live].astype(np.float64) / s[live, None].astype(np.float64))
    assert np.all(err <= 0.5 + 1e-5)


# ---------------------------------------------------------------- mixed 2/4-bit banks
MIXED = synth.Workload("mixed_small", T=12, H=256, I=128, E=8, S=1, top_k=2, group=64, twobit_frac=0.5)


def test_int2_unpack_golden_bytes():
    n = 0
    for line in open(os.path.join(GOLDEN, "int2_codes.txt")):
        f = line.split("#")[0].split()
        if not f:
            continue
        b = int(f[0], 16)
        assert [oracle.unpack2(b, p) for p in range(4)] == [int(v) for v in f[1:]], f[0]
        n += 1
    assert n >= 12


def _pack4_rows(codes):
    """int4 packing written out from the format (element 2j low nibble, 2j+1 high nibble)."""
    c = (codes.astype(np.int16) & 0xF).astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def test_int2_partials_equal_int4_partials_and_brute_force():
    rng = np.random.default_rng(21)
    rows, K, g = 24, 512, 128
    codes = rng.integers(-2, 2, size=(rows, K)).astype(np.int8)
    codes[0, :] = -2
    codes[1, :] = 1
    a = rng.integers(-127, 128, size=K).astype(np.int8)
    a[:64] = -127
    p2 = oracle.partials(a, synth.pack2_rows(codes, K // 2), g, bits=2)
    p4 = oracle.partials(a, _pack4_rows(codes), g, bits=4)
    brute = np.einsum("nqk,qk->nq", codes.astype(np.int64).reshape(rows, K // g, g),
                      a.astype(np.int64).reshape(K // g, g))
    assert np.array_equal(p2, brute) and np.array_equal(p4, brute)


def test_generator_true_2bit_bytes_unpack_to_its_codes():
    bank, c13, c2 = synth.make_bank(MIXED, with_codes=True, pack2=True)
    two = np.nonzero(bank.slot_bits == 2)[0]
    assert len(two) >= 2 and np.all(bank.slot_bits[bank.slot_bits != 2] == 4)
    assert np.array_equal(bank.slot_bits == 2, bank.twobit)
    lut = np.array([[oracle.unpack2(b, p) for p in range(4)] for b in range(256)], np.int8)
    for e in two:
        got13 = lut[bank.w13[e][:, :MIXED.H // 4]].reshape(2 * MIXED.I, MIXED.H)
        got2 = lut[bank.w2[e][:, :MIXED.I // 4]].reshape(MIXED.H, MIXED.I)
        assert np.array_equal(got13, c13[e]) and np.array_equal(got2, c2[e])
        assert not bank.w13[e][:, MIXED.H // 4:].any()  # the unused half of a 2-bit row


def test_mixed_bank_layer_equals_the_same_codes_in_int4_storage():
    tok = synth.make_tokens(MIXED)
    b4 = synth.make_bank(MIXED)
    b2 = synth.make_bank(MIXED, pack2=True)
    assert np.array_equal(b4.s13, b2.s13) and not np.array_equal(b4.w13, b2.w13)
    out4 = oracle.forward_workload(MIXED, tok, b4)
    out2 = oracle.forward_workload(MIXED, tok, b2)
    assert np.array_equal(out4, out2)
    assert np.abs(out4).max() > 0
