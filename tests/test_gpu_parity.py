"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Bit-exact: top-k ids, the permutation (counts, offsets, perm, inv) and the
int32 per-group partial sums of both projections.  Floating point: the
routing weights (fp32 vs fp64) and the layer output within the stated
tolerance (max |err| <= 2e-2 rms, 99.9% within 1e-2 rms).  The requantised
intermediate is compared code by code; a code may differ by one only where
the oracle's value sits within rounding distance of a half-step boundary
(the two sides' fp32 h differ in the last bits, the decision is the same
fp32 RNE on both).
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_router_gb300 import binding, synth

import _gpu_helpers as gh

pytestmark = pytest.mark.gpu

ALL = list(synth.WORKLOADS)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    binding._load()


def _route_gpu(w, logits):
    d = gh.dims(w)
    T, k, E = w.T, w.top_k, w.E
    dev = "cuda:0"
    out = dict(ids=torch.empty((T, k), dtype=torch.int32, device=dev),
               w=torch.empty((T, k), dtype=torch.float32, device=dev),
               counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               perm=torch.empty(T * k, dtype=torch.int32, device=dev),
               inv=torch.empty(T * k, dtype=torch.int32, device=dev))
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), dev)
    binding.moe_w4a8_route(gh.to_dev(logits), d, out["ids"], out["w"], out["counts"], out["offsets"], out["perm"],
                           out["inv"], ws)
    torch.cuda.synchronize()
    return {k_: v.cpu().numpy() for k_, v in out.items()}


def _check_route(w, logits):
    got = _route_gpu(w, logits)
    ids, wt = oracle.route(logits, w.top_k)
    counts, offsets, perm, inv = oracle.permute(ids, w.E)
    assert np.array_equal(got["ids"], ids)
    assert np.array_equal(got["counts"], counts)
    assert np.array_equal(got["offsets"], offsets)
    assert np.array_equal(got["perm"], perm)
    assert np.array_equal(got["inv"], inv)
    assert np.max(np.abs(got["w"] - wt)) < 2e-6


@pytest.mark.parametrize("name", ALL)
def test_route_bit_exact(name):
    w = synth.WORKLOADS[name]
    _check_route(w, synth.make_tokens(w).logits)


def test_route_planted_ties():
    rng = np.random.default_rng(5)
    w = synth.Workload("ties", T=300, H=256, I=128, E=64, S=0, top_k=6, group=64)
    logits = rng.integers(-2, 3, size=(w.T, w.E)).astype(np.float32)  # massive ties
    logits[rng.random(logits.shape) < 0.2] = -0.0
    logits[0, :] = 0.0
    logits[1, :] = -0.0
    _check_route(w, logits)
    w1 = synth.Workload("ties_k1", T=300, H=256, I=128, E=64, S=0, top_k=1, group=64)
    _check_route(w1, logits)
    wE = synth.Workload("ties_kE", T=50, H=256, I=128, E=32, S=0, top_k=32, group=64)
    _check_route(wE, logits[:50, :32].copy())


def test_route_nan_logits_rank_last():
    """NaN logits rank below every number (ties by index): k distinct experts per token, as the oracle."""
    rng = np.random.default_rng(9)
    w = synth.Workload("nan", T=200, H=256, I=128, E=96, S=0, top_k=7, group=64)
    logits = rng.standard_normal((w.T, w.E)).astype(np.float32)
    logits[rng.random(logits.shape) < 0.3] = np.nan
    logits[0, :] = np.nan
    logits[1, :4] = -np.inf
    logits[1, 4:] = np.nan
    got = _route_gpu(w, logits)
    ids, _ = oracle.route(logits, w.top_k)
    assert np.array_equal(got["ids"], ids)
    assert all(len(set(r)) == w.top_k for r in got["ids"].tolist())
    counts, offsets, perm, inv = oracle.permute(ids, w.E)
    assert np.array_equal(got["perm"], perm) and np.array_equal(got["inv"], inv)


def test_route_all_tokens_to_one_expert():
    w = synth.WORKLOADS["prefill_t8192"].with_tokens(3000)
    logits = synth.make_tokens(w).logits
    logits[:, 77] = 1e4
    _check_route(w, logits)


def _sample_pairs(w, tok, n, seed=0):
    """Sorted (slot, token) pairs: routed pairs of sampled tokens plus the shared slots."""
    ids, _ = oracle.route(tok.logits, w.top_k)
    rng = np.random.default_rng(seed)
    toks = gh.sample_tokens(w.T, max(1, n // (w.top_k + w.S)), seed)
    pairs = [(int(e), int(t)) for t in toks for e in ids[t]]
    pairs += [(w.E + s, int(t)) for t in toks for s in range(w.S)]
    if w.twobit_frac > 0:  # make sure 2-bit experts are covered
        tb = np.nonzero(synth.twobit_experts(w))[0]
        pairs += [(int(e), int(rng.integers(w.T))) for e in tb[:4]]
    pairs.sort()
    slots = np.array([p[0] for p in pairs], np.int32)
    tokens = np.array([p[1] for p in pairs], np.int32)
    return slots, tokens


# engine 0 = grouped mma.sync engine (any size), 1 = fused decode engine (T <= 32),
# 2 = tcgen05 engine (g a multiple of 128)
DEC_SMALL = synth.Workload("dec_small", T=8, H=2048, I=512, E=16, S=1, top_k=4, group=128)
TC_SMALL = synth.Workload("tc_small", T=300, H=256, I=128, E=8, S=1, top_k=2, group=128)
TC_ODD = synth.Workload("tc_odd", T=150, H=384, I=384, E=6, S=0, top_k=3, group=128)
TC_G256 = synth.Workload("tc_g256", T=140, H=512, I=256, E=4, S=1, top_k=2, group=256)
DEC_G64 = synth.Workload("dec_g64", T=6, H=2048, I=512, E=8, S=1, top_k=3, group=64)
EXTRA = {w.name: w for w in (DEC_SMALL, TC_SMALL, TC_ODD, TC_G256, DEC_G64)}
PARTIALS_CASES = ([(n, 0) for n in ALL] + [("decode_t4", 1), ("decode_verify_t12", 1), ("dec_small", 1), ("dec_g64", 1)] +
                  [(n, 2) for n in ("prefill_t8192", "large_bank_t2048", "decode_t4", "tc_small", "tc_odd",
                                    "tc_g256")])


def _workload(name):
    return EXTRA[name] if name in EXTRA else synth.WORKLOADS[name]


@pytest.mark.parametrize("name,engine", PARTIALS_CASES)
def test_gemm1_partials_bit_exact(name, engine):
    w = _workload(name)
    tok = synth.make_tokens(w)
    bank = gh.bank_of(w)
    w13, _, _, _ = gh.device_bank(w)
    slots, tokens = _sample_pairs(w, tok, 96)
    d = gh.dims(w)
    n = slots.shape[0]
    p1 = torch.empty((n, 2 * w.I, w.H // w.group), dtype=torch.int32, device="cuda:0")
    ws = binding.alloc_workspace(binding.partials_workspace_size(d, n), "cuda:0")
    binding.moe_w4a8_gemm1_partials(gh.to_dev(tok.x_q), w13, d, gh.to_dev(tokens), gh.to_dev(slots), p1, ws, engine)
    torch.cuda.synchronize()
    got = p1.cpu().numpy()
    for r in range(n):
        ref = oracle.partials(tok.x_q[tokens[r]], bank.w13[slots[r]], w.group)
        bad = np.argwhere(got[r] != ref)
        assert bad.size == 0, (f"pair {r}: token {tokens[r]} slot {slots[r]}: {len(bad)} of {ref.size} differ, "
                               f"first (row, group) {bad[:6].tolist()}")


@pytest.mark.parametrize("name,engine", PARTIALS_CASES)
def test_gemm2_partials_bit_exact(name, engine):
    w = _workload(name)
    tok = synth.make_tokens(w)
    bank = gh.bank_of(w)
    _, _, w2, _ = gh.device_bank(w)
    slots, _ = _sample_pairs(w, tok, 96, seed=1)
    n = slots.shape[0]
    rng = np.random.default_rng(2)
    h_q = rng.integers(-127, 128, size=(n, w.I)).astype(np.int8)
    h_q[0, :] = 127
    if n > 1:
        h_q[1, :] = -127
    d = gh.dims(w)
    p2 = torch.empty((n, w.H, w.I // w.group), dtype=torch.int32, device="cuda:0")
    ws = binding.alloc_workspace(binding.partials_workspace_size(d, n), "cuda:0")
    binding.moe_w4a8_gemm2_partials(gh.to_dev(h_q), w2, d, gh.to_dev(slots), p2, ws, engine)
    torch.cuda.synchronize()
    got = p2.cpu().numpy()
    for r in range(n):
        ref = oracle.partials(h_q[r], bank.w2[slots[r]], w.group)
        bad = np.argwhere(got[r] != ref)
        assert bad.size == 0, f"pair {r}: slot {slots[r]}: {len(bad)} of {ref.size} differ, first {bad[:6].tolist()}"


@pytest.mark.parametrize("name", ALL)
def test_forward_matches_oracle(name):
    w = synth.WORKLOADS[name]
    tok = synth.make_tokens(w)
    bank = gh.bank_of(w)
    out = gh.run_forward(w, tok)
    sel = gh.sample_tokens(w.T, 48)
    if w.T > 48:
        # plus every token routed to the ten least-loaded touched experts (the skewed tail's partial tiles)
        ids, _ = oracle.route(tok.logits, w.top_k)
        counts = np.bincount(ids.ravel(), minlength=w.E)
        tail = [e for e in np.argsort(counts, kind="stable") if counts[e] > 0][:10]
        extra = np.nonzero(np.isin(ids, tail).any(axis=1))[0]
        sel = np.union1d(sel, extra)
    ref = gh.oracle_out(w, tok, bank, sel)
    gh.assert_output_close(out[sel], ref, name)
    assert np.all(np.isfinite(out))
    again = gh.run_forward(w, tok)
    assert np.array_equal(out, again), "two runs differ"


@pytest.mark.parametrize("name,engine", [("tiny", -1), ("decode_t4", 0), ("decode_t4", 1),
                                         ("decode_verify_t12", 0), ("decode_verify_t12", 1), ("dec_small", 1),
                                         ("decode_t4", 2), ("tc_small", 2), ("tc_odd", 2), ("tc_g256", 2)])
def test_requantised_intermediate(name, engine):
    w = _workload(name)
    tok = synth.make_tokens(w)
    bank = gh.bank_of(w)
    w13, s13, w2, s2 = gh.device_bank(w)
    d = gh.dims(w)
    P = w.T * (w.top_k + w.S)
    out = torch.empty((w.T, w.H), dtype=torch.float32, device="cuda:0")
    h_q = torch.empty((P, w.I), dtype=torch.int8, device="cuda:0")
    s_h = torch.empty(P, dtype=torch.float32, device="cuda:0")
    y = torch.empty((P, w.H), dtype=torch.float32, device="cuda:0")
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    binding.moe_w4a8_forward_debug(gh.to_dev(tok.x_q), gh.to_dev(tok.x_scale), gh.to_dev(tok.logits), w13, s13, w2,
                                   s2, d, out, ws, h_q, s_h, y, engine=engine)
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    ref_out = gh.oracle_out(w, tok, bank)
    gh.assert_output_close(out.cpu().numpy(), ref_out, f"{name} engine {engine}")
    h_q, s_h, y = h_q.cpu().numpy(), s_h.cpu().numpy(), y.cpu().numpy()
    ids, _ = oracle.route(tok.logits, w.top_k)
    _, _, _, inv = oracle.permute(ids, w.E)
    od = oracle.dims(w.T, w.H, w.I, w.E, w.S, w.top_k, w.group)
    flips = 0
    for t in range(w.T):
        rows = [(int(inv[t * w.top_k + j]), int(ids[t, j])) for j in range(w.top_k)]
        rows += [(w.T * w.top_k + s * w.T + t, w.E + s) for s in range(w.S)]
        for row, slot in rows:
            hq_ref, sh_ref, y_ref = oracle.pair_output(od, tok.x_q, tok.x_scale, bank.w13, bank.s13, bank.w2,
                                                       bank.s2, t, slot)
            assert abs(s_h[row] - sh_ref) <= 1e-5 * sh_ref
            diff = h_q[row].astype(int) - hq_ref.astype(int)
            assert np.all(np.abs(diff) <= 1)
            if diff.any():
                # only at half-step boundaries of the oracle's own value
                _, _, h = oracle.hidden(tok.x_q[t], tok.x_scale[t], bank.w13[slot], bank.s13[slot], w.group)
                frac = np.abs(np.abs(h[diff != 0] / sh_ref) % 1.0 - 0.5)
                assert np.all(frac < 1e-3), frac
                flips += int(np.count_nonzero(diff))
            scale = np.max(np.abs(y_ref)) + 1e-30
            assert np.max(np.abs(y[row] - y_ref)) <= 2e-2 * scale
    assert flips <= 1e-3 * P * w.I


# ------------------------------------------------------------------ edge cases

SMALL = synth.Workload("small_s1", T=16, H=256, I=128, E=8, S=1, top_k=2, group=64)


@pytest.mark.parametrize("T", [1, 2, 37, 64, 65, 130, 257])
def test_ragged_batch_sizes(T):
    w = SMALL.with_tokens(T)
    tok = synth.make_tokens(w)
    out = gh.run_forward(w, tok)
    gh.assert_output_close(out, gh.oracle_out(w, tok, gh.bank_of(w)), f"T={T}")


@pytest.mark.parametrize("k", [1, 8])
def test_top_k_extremes(k):
    w = synth.Workload("k", T=40, H=256, I=128, E=8, S=0, top_k=k, group=64)
    tok = synth.make_tokens(w)
    gh.assert_output_close(gh.run_forward(w, tok), gh.oracle_out(w, tok, gh.bank_of(w)), f"k={k}")


def test_single_expert_dense_case():
    w = synth.Workload("dense", T=70, H=256, I=128, E=1, S=0, top_k=1, group=128)
    tok = synth.make_tokens(w)
    gh.assert_output_close(gh.run_forward(w, tok), gh.oracle_out(w, tok, gh.bank_of(w)), "E=1")


def test_all_tokens_on_one_expert_spans_many_tiles():
    w = SMALL.with_tokens(300)
    tok = synth.make_tokens(w)
    tok.logits[:, 5] = 50.0
    out = gh.run_forward(w, tok)
    gh.assert_output_close(out, gh.oracle_out(w, tok, gh.bank_of(w)), "one hot expert")


def test_zero_weight_expert_and_zero_token():
    w = SMALL.with_tokens(33)
    tok = synth.make_tokens(w)
    b = gh.bank_of(w)
    bank = synth.Bank(b.w13.copy(), b.s13.copy(), b.w2.copy(), b.s2.copy(), b.twobit)
    for a in (bank.w13, bank.s13, bank.w2, bank.s2):
        a[3] = 0
    tok.x_q[4] = 0
    tok.x_scale[4] = 0.0
    dev_bank = tuple(gh.to_dev(a) for a in (bank.w13, bank.s13, bank.w2, bank.s2))
    out = gh.run_forward(w, tok, dev_bank)
    ref = gh.oracle_out(w, tok, bank)
    gh.assert_output_close(out, ref, "zero expert")
    assert np.array_equal(out[4], np.zeros(w.H, np.float32))  # zero activations give exactly zero


def test_empty_batch_leaves_output_untouched():
    w = SMALL.with_tokens(0)
    w13, s13, w2, s2 = gh.device_bank(w)
    d = gh.dims(w)
    out = torch.empty((0, w.H), dtype=torch.float32, device="cuda:0")
    e = lambda *s, dt=torch.float32: torch.empty(s, dtype=dt, device="cuda:0")  # noqa: E731
    ws = binding.alloc_workspace(256, "cuda:0")
    binding.moe_w4a8_forward(e(0, w.H, dt=torch.int8), e(0), e(0, w.E), w13, s13, w2, s2, d, out, ws)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ fused decode engine

def _forward_engine(w, tok, engine, bank_dev=None):
    w13, s13, w2, s2 = bank_dev if bank_dev is not None else gh.device_bank(w)
    d = gh.dims(w)
    out = torch.full((w.T, w.H), float("nan"), dtype=torch.float32, device="cuda:0")
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    binding.moe_w4a8_forward_debug(gh.to_dev(tok.x_q), gh.to_dev(tok.x_scale), gh.to_dev(tok.logits), w13, s13, w2,
                                   s2, d, out, ws, engine=engine)
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("T", [1, 2, 3, 17, 32])
def test_decode_engine_ragged_batches(T):
    w = DEC_SMALL.with_tokens(T)
    tok = synth.make_tokens(w)
    out = _forward_engine(w, tok, 1)
    gh.assert_output_close(out, gh.oracle_out(w, tok, gh.bank_of(w)), f"decode T={T}")


@pytest.mark.parametrize("k,S", [(1, 0), (16, 1), (4, 0), (4, 2)])
def test_decode_engine_top_k_and_shared(k, S):
    w = synth.Workload("dk", T=9, H=2048, I=512, E=16, S=S, top_k=k, group=64)
    tok = synth.make_tokens(w)
    out = _forward_engine(w, tok, 1)
    gh.assert_output_close(out, gh.oracle_out(w, tok, gh.bank_of(w)), f"decode k={k} S={S}")


@pytest.mark.parametrize("E", [64, 600])
def test_decode_engine_routes_planted_ties(E):
    """The fused kernel's own routing on massively tied logits (E > 512 takes its wide path)."""
    w = synth.Workload("dties", T=12, H=2048, I=512, E=E, S=1, top_k=6, group=128)
    tok = synth.make_tokens(w)
    rng = np.random.default_rng(7)
    lg = rng.integers(-2, 3, size=(w.T, w.E)).astype(np.float32)
    lg[rng.random(lg.shape) < 0.2] = -0.0
    lg[0, :] = 0.0
    lg[1, :] = -0.0
    tok.logits[...] = lg
    out = _forward_engine(w, tok, 1)
    gh.assert_output_close(out, gh.oracle_out(w, tok, gh.bank_of(w)), f"decode ties E={E}")


def _debug_routing(w, tok, engine):
    """Runs moe_w4a8_forward_debug on `engine` and reads back the routing it used."""
    w13, s13, w2, s2 = gh.device_bank(w)
    d = gh.dims(w)
    dev = "cuda:0"
    out = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), dev)
    binding.moe_w4a8_forward_debug(gh.to_dev(tok.x_q), gh.to_dev(tok.x_scale), gh.to_dev(tok.logits), w13, s13, w2,
                                   s2, d, out, ws, engine=engine)
    got = dict(ids=torch.empty((w.T, w.top_k), dtype=torch.int32, device=dev),
               w=torch.empty((w.T, w.top_k), dtype=torch.float32, device=dev),
               perm=torch.empty(w.T * w.top_k, dtype=torch.int32, device=dev),
               inv=torch.empty(w.T * w.top_k, dtype=torch.int32, device=dev))
    binding.moe_w4a8_debug_routing(d, ws, got["ids"], got["w"], got["perm"], got["inv"])
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    return {k_: v.cpu().numpy() for k_, v in got.items()}


@pytest.mark.parametrize("name,engine", [("decode_t4", 1), ("decode_verify_t12", 1), ("dec_small", 1),
                                         ("decode_t4", 0), ("tc_small", 2)])
def test_engine_routing_is_the_oracles(name, engine):
    """The routing each engine used inside the layer call (the decode kernel's own in-kernel top-k and pair
    sort included): ids, permutation and inverse bit-exact against the oracle, weights within 2e-6."""
    w = _workload(name)
    tok = synth.make_tokens(w)
    got = _debug_routing(w, tok, engine)
    ids, wt = oracle.route(tok.logits, w.top_k)
    _, _, perm, inv = oracle.permute(ids, w.E)
    assert np.array_equal(got["ids"], ids)
    assert np.array_equal(got["perm"], perm)
    assert np.array_equal(got["inv"], inv)
    assert np.max(np.abs(got["w"] - wt)) < 2e-6


@pytest.mark.parametrize("E", [64, 600])
def test_decode_engine_routing_of_planted_ties_is_the_oracles(E):
    """Massively tied and signed-zero logits through the decode kernel's own routing (E > 512 takes its
    wide path): ids and permutation bit-exact."""
    w = synth.Workload("dties", T=12, H=2048, I=512, E=E, S=1, top_k=6, group=128)
    tok = synth.make_tokens(w)
    rng = np.random.default_rng(7)
    lg = rng.integers(-2, 3, size=(w.T, w.E)).astype(np.float32)
    lg[rng.random(lg.shape) < 0.2] = -0.0
    lg[0, :] = 0.0
    lg[1, :] = -0.0
    tok.logits[...] = lg
    got = _debug_routing(w, tok, 1)
    ids, wt = oracle.route(tok.logits, w.top_k)
    _, _, perm, inv = oracle.permute(ids, w.E)
    assert np.array_equal(got["ids"], ids)
    assert np.array_equal(got["perm"], perm)
    assert np.array_equal(got["inv"], inv)
    assert np.max(np.abs(got["w"] - wt)) < 2e-6


def test_decode_engine_ranks_nan_logits_last():
    """NaN logits in the decode kernel's own routing: never chosen while k numbers remain, so those tokens
    match the oracle; a token whose logits are all NaN gets the lowest k experts (NaN weights, NaN output)."""
    w = synth.Workload("dnan", T=10, H=2048, I=512, E=64, S=1, top_k=6, group=128)
    tok = synth.make_tokens(w)
    orig = tok.logits.copy()
    rng = np.random.default_rng(3)
    tok.logits[rng.random(tok.logits.shape) < 0.4] = np.nan
    tok.logits[2, :] = np.nan
    tok.logits[3, :58] = np.nan  # exactly k numbers left
    tok.logits[3, 58:] = orig[3, 58:]
    assert all(np.count_nonzero(~np.isnan(tok.logits[t])) >= w.top_k for t in range(w.T) if t != 2)
    out = _forward_engine(w, tok, 1)
    ref = gh.oracle_out(w, tok, gh.bank_of(w))
    ok = [t for t in range(w.T) if t != 2]
    gh.assert_output_close(out[ok], ref[ok], "decode engine, NaN logits")
    assert np.all(np.isnan(out[2])) and np.all(np.isnan(ref[2]))
    ids, _ = oracle.route(tok.logits, w.top_k)
    assert ids[2].tolist() == list(range(w.top_k)) and ids[3].tolist() == sorted(ids[3].tolist(), key=lambda e: -tok.logits[3, e])


def test_decode_engine_matches_grouped_engine_on_large_bank_shape():
    w = synth.WORKLOADS["large_bank_t2048"].with_tokens(6)
    tok = synth.make_tokens(w)
    a = _forward_engine(w, tok, 1)
    b = _forward_engine(w, tok, 0)
    ref = gh.oracle_out(w, tok, gh.bank_of(w))
    gh.assert_output_close(a, ref, "decode engine, large bank")
    gh.assert_output_close(b, ref, "grouped engine, large bank")


@pytest.mark.parametrize("H,I,T", [(2048, 1024, 5), (4096, 2048, 3), (2048, 2048, 9)])
def test_decode_engine_intermediate_widths(H, I, T):
    """The decode engine at intermediate widths I = 1024 and 2048 (both hidden sizes): auto-selected, and
    within tolerance of the oracle, with a 2-bit-free and a mixed bank (the latter through the uniform and
    the compact storage, bit for bit alike)."""
    w = synth.Workload(f"dec_h{H}_i{I}", T=T, H=H, I=I, E=40, S=1, top_k=4, group=128, twobit_frac=0.25)
    assert binding.moe_w4a8_engine_for(gh.dims(w)) == 1
    tok = synth.make_tokens(w)
    got = _forward_engine(w, tok, 1)
    gh.assert_output_close(got, gh.oracle_out(w, tok, gh.bank_of(w)), f"decode engine H={H} I={I}")
    b2 = synth.make_bank(w, pack2=True)
    d = gh.dims(w)
    x = [gh.to_dev(a) for a in (tok.x_q, tok.x_scale, tok.logits)]
    s13, s2, bits = gh.to_dev(b2.s13), gh.to_dev(b2.s2), gh.to_dev(b2.slot_bits)
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    out = torch.empty((w.T, w.H), dtype=torch.float32, device="cuda:0")
    binding.moe_w4a8_forward_w2w4(*x, gh.to_dev(b2.w13), s13, gh.to_dev(b2.w2), s2, bits, d, out, ws)
    w13c, o13, w2c, o2 = synth.compact_bank(b2)
    outc = torch.full_like(out, float("nan"))
    binding.moe_w4a8_forward_w2w4_compact(*x, gh.to_dev(w13c), gh.to_dev(o13), s13, gh.to_dev(w2c), gh.to_dev(o2),
                                          s2, bits, d, outc, ws)
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    mixed = out.cpu().numpy()
    gh.assert_output_close(mixed, oracle.forward_workload(w, tok, b2), f"decode engine H={H} I={I}, mixed bank")
    assert np.array_equal(outc.cpu().numpy(), mixed)


def test_decode_engine_is_deterministic_and_auto_selected():
    w = synth.WORKLOADS["decode_t4"]
    tok = synth.make_tokens(w, batch=3)
    a = _forward_engine(w, tok, 1)
    b = _forward_engine(w, tok, -1)
    assert np.array_equal(a, b)


def test_decode_engine_rejects_batches_beyond_its_limits():
    w = DEC_SMALL.with_tokens(33)
    tok = synth.make_tokens(w)
    with pytest.raises(binding.MoeError) as e:
        _forward_engine(w, tok, 1)
    assert e.value.status == 2


def test_bounded_wait_reports_timeout_and_context_survives():
    w = synth.WORKLOADS["decode_t4"]
    d = gh.dims(w)
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    binding.moe_w4a8_selftest_barrier_timeout(ws)
    assert binding.moe_w4a8_device_status(ws) == 5
    # the same workspace and context serve a normal call afterwards
    tok = synth.make_tokens(w)
    w13, s13, w2, s2 = gh.device_bank(w)
    out = torch.empty((w.T, w.H), dtype=torch.float32, device="cuda:0")
    binding.moe_w4a8_forward(gh.to_dev(tok.x_q), gh.to_dev(tok.x_scale), gh.to_dev(tok.logits), w13, s13, w2, s2, d,
                             out, ws)
    assert binding.moe_w4a8_device_status(ws) == 0
    gh.assert_output_close(out.cpu().numpy(), gh.oracle_out(w, tok, gh.bank_of(w)), "after timeout")


# ------------------------------------------------------------------ tcgen05 engine

@pytest.mark.parametrize("T", [1, 2, 37, 129, 300])
def test_tcgen05_engine_ragged_batches(T):
    w = TC_SMALL.with_tokens(T)
    tok = synth.make_tokens(w)
    out = _forward_engine(w, tok, 2)
    gh.assert_output_close(out, gh.oracle_out(w, tok, gh.bank_of(w)), f"tcgen05 T={T}")


@pytest.mark.parametrize("name", ["tc_odd", "tc_g256"])
def test_tcgen05_engine_shapes(name):
    w = EXTRA[name]
    tok = synth.make_tokens(w)
    out = _forward_engine(w, tok, 2)
    gh.assert_output_close(out, gh.oracle_out(w, tok, gh.bank_of(w)), name)


def test_tcgen05_engine_one_expert_spans_many_token_tiles():
    w = TC_SMALL.with_tokens(700)
    tok = synth.make_tokens(w)
    tok.logits[:, 5] = 50.0
    out = _forward_engine(w, tok, 2)
    gh.assert_output_close(out, gh.oracle_out(w, tok, gh.bank_of(w)), "one hot expert")


def test_tcgen05_engine_matches_grouped_engine_on_large_bank():
    w = synth.WORKLOADS["large_bank_t2048"].with_tokens(200)
    tok = synth.make_tokens(w)
    a = _forward_engine(w, tok, 2)
    b = _forward_engine(w, tok, 0)
    sel = gh.sample_tokens(w.T, 24)
    ref = gh.oracle_out(w, tok, gh.bank_of(w), sel)
    gh.assert_output_close(a[sel], ref, "tcgen05 engine, large bank")
    gh.assert_output_close(b[sel], ref, "grouped engine, large bank")
    again = _forward_engine(w, tok, 2)
    assert np.array_equal(a, again), "two runs differ"


def test_tcgen05_engine_is_auto_selected_for_large_batches():
    assert binding.moe_w4a8_engine_for(gh.dims(synth.WORKLOADS["prefill_t8192"])) == 2
    assert binding.moe_w4a8_engine_for(gh.dims(synth.WORKLOADS["large_bank_t2048"])) == 2
    assert binding.moe_w4a8_engine_for(gh.dims(synth.WORKLOADS["decode_t4"])) == 1
    assert binding.moe_w4a8_engine_for(gh.dims(synth.WORKLOADS["tiny"])) == 0  # g = 64


def test_tcgen05_engine_rejects_groups_it_does_not_tile():
    w = SMALL.with_tokens(8)  # g = 64
    tok = synth.make_tokens(w)
    with pytest.raises(binding.MoeError) as e:
        _forward_engine(w, tok, 2)
    assert e.value.status == 2


@pytest.mark.parametrize("name,pinned_in,pinned_out", [("decode_t4", True, True), ("decode_t4", False, False),
                                                       ("decode_t4", True, False), ("tc_small", True, True),
                                                       ("small_s1", False, True)])
def test_forward_host_buffers_match_device_forward(name, pinned_in, pinned_out):
    """Host-resident activations/logits/output: the same kernels, so the same bits as the device call."""
    w = _workload(name) if name in EXTRA else (SMALL if name == "small_s1" else synth.WORKLOADS[name])
    tok = synth.make_tokens(w)
    d = gh.dims(w)
    w13, s13, w2, s2 = gh.device_bank(w)
    ws = binding.alloc_workspace(binding.moe_w4a8_forward_host_workspace_size(d), "cuda:0")
    dev_out = torch.empty((w.T, w.H), dtype=torch.float32, device="cuda:0")
    binding.moe_w4a8_forward(gh.to_dev(tok.x_q), gh.to_dev(tok.x_scale), gh.to_dev(tok.logits), w13, s13, w2, s2, d,
                             dev_out, ws)
    host_in = [torch.from_numpy(a.copy()) for a in (tok.x_q, tok.x_scale, tok.logits)]
    if pinned_in:
        host_in = [t.pin_memory() for t in host_in]
    host_out = torch.full((w.T, w.H), float("nan"), dtype=torch.float32)
    if pinned_out:
        host_out = host_out.pin_memory()
    binding.moe_w4a8_forward_host(*host_in, w13, s13, w2, s2, d, host_out, ws)
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    assert torch.equal(host_out, dev_out.cpu())


@pytest.mark.parametrize("name", ["decode_t4", "decode_verify_t12", "dec_small", "dec_g64", "large_bank_t2048",
                                  "tc_small", "small_s1"])
def test_forward_bf16_quantises_on_device_bit_exactly(name):
    """S0 on the device: the same codes as the oracle's S0, so the same output bits as moe_w4a8_forward."""
    if name == "small_s1":
        w = SMALL
    elif name == "large_bank_t2048":
        w = synth.WORKLOADS[name].with_tokens(6)  # the decode engine at H = 4096
    else:
        w = _workload(name)
    xb = synth.bf16_activations(w)
    xb[0, :] = 0.0                      # an all-zero token: s = 0, codes 0
    if w.T > 1:
        xb[1, 5] = -3.0 * np.abs(xb[1]).max()  # the row maximum at a negative value
    bits = (np.ascontiguousarray(xb, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x_q, x_scale = oracle.quantize_bf16(bits)
    assert x_scale[0] == 0 and not x_q[0].any()
    tok = synth.make_tokens(w)
    d = gh.dims(w)
    w13, s13, w2, s2 = gh.device_bank(w)
    ws = binding.alloc_workspace(binding.moe_w4a8_forward_bf16_workspace_size(d), "cuda:0")
    ref = torch.empty((w.T, w.H), dtype=torch.float32, device="cuda:0")
    binding.moe_w4a8_forward(gh.to_dev(x_q), gh.to_dev(x_scale), gh.to_dev(tok.logits), w13, s13, w2, s2, d, ref, ws)
    out = torch.full((w.T, w.H), float("nan"), dtype=torch.float32, device="cuda:0")
    x_dev = torch.from_numpy(bits.view(np.int16)).to("cuda:0").view(torch.bfloat16)
    binding.moe_w4a8_forward_bf16(x_dev, gh.to_dev(tok.logits), w13, s13, w2, s2, d, out, ws)
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("name", ["decode_t4", "tc_small"])
def test_layer_call_captures_into_a_cuda_graph(name):
    """The call enqueues kernels only (no sync, no allocation): a captured graph replays it on new inputs."""
    w = _workload(name) if name in EXTRA else synth.WORKLOADS[name]
    d = gh.dims(w)
    w13, s13, w2, s2 = gh.device_bank(w)
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    toks = [synth.make_tokens(w, batch=b) for b in range(3)]
    x_q, x_s, lg = (gh.to_dev(a) for a in (toks[0].x_q, toks[0].x_scale, toks[0].logits))
    out = torch.empty((w.T, w.H), dtype=torch.float32, device="cuda:0")
    eager = []
    for t in toks:
        o = torch.empty_like(out)
        binding.moe_w4a8_forward(gh.to_dev(t.x_q), gh.to_dev(t.x_scale), gh.to_dev(t.logits), w13, s13, w2, s2, d, o, ws)
        eager.append(o)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            binding.moe_w4a8_forward(x_q, x_s, lg, w13, s13, w2, s2, d, out, ws)
    for b in (1, 2, 0):
        x_q.copy_(gh.to_dev(toks[b].x_q))
        x_s.copy_(gh.to_dev(toks[b].x_scale))
        lg.copy_(gh.to_dev(toks[b].logits))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager[b]), f"replay on batch {b}"
    assert binding.moe_w4a8_device_status(ws) == 0


DEC_MIXED = synth.Workload("dec_mixed", T=8, H=2048, I=512, E=32, S=1, top_k=4, group=128, twobit_frac=0.5)


@pytest.mark.parametrize("name", ["dec_mixed", "large_bank_t2048"])
def test_mixed_2bit_bank_on_the_decode_engine(name):
    """True 2-bit packing of the bank's 2-bit experts: against the oracle, and against the same codes
    stored as int4 (only the fp32 fold order differs between the two paths)."""
    w = DEC_MIXED if name == "dec_mixed" else synth.WORKLOADS[name].with_tokens(6)
    tok = synth.make_tokens(w)
    b2 = synth.make_bank(w, pack2=True)
    assert (b2.slot_bits == 2).sum() >= 2
    d = gh.dims(w)
    dev = [gh.to_dev(a) for a in (b2.w13, b2.s13, b2.w2, b2.s2)]
    bits = gh.to_dev(b2.slot_bits)
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    x = [gh.to_dev(a) for a in (tok.x_q, tok.x_scale, tok.logits)]
    out = torch.empty((w.T, w.H), dtype=torch.float32, device="cuda:0")
    binding.moe_w4a8_forward_w2w4(*x, *dev, bits, d, out, ws)
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    got = out.cpu().numpy()
    gh.assert_output_close(got, oracle.forward_workload(w, tok, b2), f"mixed bank {name}")
    # the same codes in int4 storage through the int4 path
    w13, s13, w2, s2 = gh.device_bank(w)
    ref = torch.empty_like(out)
    binding.moe_w4a8_forward(*x, w13, s13, w2, s2, d, ref, ws)
    ref = ref.cpu().numpy()
    rms = np.sqrt(np.mean(ref.astype(np.float64) ** 2))
    # fp32 fold order only (and, rarely, a requantisation code one step apart at a half-step)
    assert np.max(np.abs(got - ref)) <= 1e-3 * rms
    # every slot 4-bit: the int4 path itself, bit for bit
    all4 = torch.full((w.E + w.S,), 4, dtype=torch.uint8, device="cuda:0")
    binding.moe_w4a8_forward_w2w4(*x, w13, s13, w2, s2, all4, d, out, ws)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref)


TC_MIXED = synth.Workload("tc_mixed", T=400, H=512, I=256, E=8, S=1, top_k=2, group=128, twobit_frac=0.5)


@pytest.mark.parametrize("name", ["tc_mixed", "large_bank_t2048"])
def test_mixed_2bit_bank_on_the_tcgen05_engine(name):
    """A mixed 2/4-bit bank on the tcgen05 engine (batches past the decode engine's range): against the
    oracle (every token of the small case; for the 2048-token large bank the 48 sampled tokens plus those
    routed to the least-loaded experts), against the same codes in int4 storage, and bit for bit against
    the int4 path when every slot is 4-bit."""
    w = TC_MIXED if name == "tc_mixed" else synth.WORKLOADS[name]
    tok = synth.make_tokens(w)
    b2 = synth.make_bank(w, pack2=True)
    assert (b2.slot_bits == 2).sum() >= 2
    d = gh.dims(w)
    assert binding.moe_w4a8_engine_for(d) == 2
    dev = [gh.to_dev(a) for a in (b2.w13, b2.s13, b2.w2, b2.s2)]
    bits = gh.to_dev(b2.slot_bits)
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    x = [gh.to_dev(a) for a in (tok.x_q, tok.x_scale, tok.logits)]
    out = torch.empty((w.T, w.H), dtype=torch.float32, device="cuda:0")
    binding.moe_w4a8_forward_w2w4(*x, *dev, bits, d, out, ws)
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    got = out.cpu().numpy()
    sel = np.arange(w.T) if w.T <= 400 else gh.sample_tokens(w.T, 48)
    if w.T > 400:
        ids, _ = oracle.route(tok.logits, w.top_k)
        counts = np.bincount(ids.ravel(), minlength=w.E)
        tail = [e for e in np.argsort(counts, kind="stable") if counts[e] > 0][:6]
        sel = np.union1d(sel, np.nonzero(np.isin(ids, tail).any(axis=1))[0][:48])
    gh.assert_output_close(got[sel], oracle.forward_workload(w, tok, b2, sel), f"mixed bank {name} (tcgen05)")
    # the same codes in int4 storage through the int4 path of the same engine
    w13, s13, w2, s2 = gh.device_bank(w)
    ref = torch.empty_like(out)
    binding.moe_w4a8_forward(*x, w13, s13, w2, s2, d, ref, ws)
    ref = ref.cpu().numpy()
    rms = np.sqrt(np.mean(ref.astype(np.float64) ** 2))
    # the same integer products; only a requantisation code one step apart at a half-step can differ
    assert np.max(np.abs(got - ref)) <= 1e-3 * rms
    all4 = torch.full((w.E + w.S,), 4, dtype=torch.uint8, device="cuda:0")
    binding.moe_w4a8_forward_w2w4(*x, w13, s13, w2, s2, all4, d, out, ws)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref)


@pytest.mark.parametrize("name,T", [("dec_mixed", None), ("tc_mixed", None), ("large_bank_t2048", 6),
                                    ("large_bank_t2048", None)])
def test_compact_mixed_bank_reproduces_the_uniform_layout(name, T):
    """Compact storage of a mixed 2/4-bit bank (each slot's rows at its own width, slots back to back, the
    library's layout helper giving the offsets): bit for bit the output of the uniform layout on the same
    codes -- on the decode engine (dec_mixed, 6 tokens of the large bank) and the tcgen05 engine (tc_mixed,
    the 2048-token large bank) -- so the oracle checks of the uniform layout carry over; the small case is
    also checked against the oracle directly."""
    w = {"dec_mixed": DEC_MIXED, "tc_mixed": TC_MIXED}.get(name) or synth.WORKLOADS[name]
    if T is not None:
        w = w.with_tokens(T)
    tok = synth.make_tokens(w)
    b2 = synth.make_bank(w, pack2=True)
    assert (b2.slot_bits == 2).sum() >= 2
    d = gh.dims(w)
    w13c, o13, w2c, o2 = synth.compact_bank(b2)
    l13, l2, n13, n2 = binding.moe_w4a8_mixed_bank_layout(torch.from_numpy(b2.slot_bits.copy()), d)
    assert np.array_equal(l13.numpy(), o13) and np.array_equal(l2.numpy(), o2) and (n13, n2) == (w13c.size, w2c.size)
    assert w13c.size < b2.w13.size and w2c.size < b2.w2.size
    x = [gh.to_dev(a) for a in (tok.x_q, tok.x_scale, tok.logits)]
    s13, s2, bits = gh.to_dev(b2.s13), gh.to_dev(b2.s2), gh.to_dev(b2.slot_bits)
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    ref = torch.empty((w.T, w.H), dtype=torch.float32, device="cuda:0")
    binding.moe_w4a8_forward_w2w4(*x, gh.to_dev(b2.w13), s13, gh.to_dev(b2.w2), s2, bits, d, ref, ws)
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    out = torch.full_like(ref, float("nan"))
    binding.moe_w4a8_forward_w2w4_compact(*x, gh.to_dev(w13c), gh.to_dev(o13), s13, gh.to_dev(w2c), gh.to_dev(o2),
                                          s2, bits, d, out, ws)
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    got = out.cpu().numpy()
    assert np.array_equal(got, ref.cpu().numpy())
    if w.T <= 8:
        gh.assert_output_close(got, oracle.forward_workload(w, tok, b2), f"compact mixed bank {name}")


def _routed_call(w, tok, ids, wts):
    w13, s13, w2, s2 = gh.device_bank(w)
    d = gh.dims(w)
    out = torch.empty((w.T, w.H), dtype=torch.float32, device="cuda:0")
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    binding.moe_w4a8_forward_routed(gh.to_dev(tok.x_q), gh.to_dev(tok.x_scale), gh.to_dev(ids.astype(np.int32)),
                                    gh.to_dev(wts.astype(np.float32)), w13, s13, w2, s2, d, out, ws)
    torch.cuda.synchronize()
    assert binding.moe_w4a8_device_status(ws) == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("name,engine", [("decode_t4", 1), ("decode_verify_t12", 1), ("tc_small", 2), ("tiny", 0)])
def test_supplied_routing_reproduces_the_layer(name, engine):
    """A routing cache hit: the routing a layer call computed, handed back through moe_w4a8_forward_routed,
    gives that call's output bit for bit (each engine, its own routing); the oracle's routing gives the
    oracle's output within the stated tolerance."""
    w = _workload(name)
    tok = synth.make_tokens(w)
    assert binding.moe_w4a8_engine_for(gh.dims(w)) == engine
    got = _debug_routing(w, tok, engine)
    ref = _forward_engine(w, tok, engine)
    out = _routed_call(w, tok, got["ids"], got["w"])
    assert np.array_equal(out, ref)
    ids, wt = oracle.route(tok.logits, w.top_k)
    out_o = _routed_call(w, tok, ids, wt)
    sel = gh.sample_tokens(w.T, 48)
    gh.assert_output_close(out_o[sel], gh.oracle_out(w, tok, gh.bank_of(w), sel), f"{name} oracle routing supplied")


@pytest.mark.parametrize("name", ["dec_small", "tc_small"])
def test_supplied_routing_with_repeats_and_out_of_range_ids(name):
    """Ids outside [0, E) are clamped and a token may name an expert twice: every pair is computed and
    weighted as given (against the oracle's per-pair outputs summed in the same order)."""
    w = _workload(name)
    tok = synth.make_tokens(w)
    rng = np.random.default_rng(3)
    ids = rng.integers(0, w.E, size=(w.T, w.top_k)).astype(np.int64)
    ids[0, :] = ids[0, 0]                      # one expert, k times
    ids[1, 0] = -5
    ids[1, -1] = w.E + 7
    wts = rng.random((w.T, w.top_k)).astype(np.float32)
    out = _routed_call(w, tok, ids, wts)
    assert np.all(np.isfinite(out))
    bank = gh.bank_of(w)
    od = oracle.dims(w.T, w.H, w.I, w.E, w.S, w.top_k, w.group)
    clamped = np.clip(ids, 0, w.E - 1)
    for t in gh.sample_tokens(w.T, 12):
        ref = np.zeros(w.H)
        for j in range(w.top_k):
            _, _, y = oracle.pair_output(od, tok.x_q, tok.x_scale, bank.w13, bank.s13, bank.w2, bank.s2, t,
                                         int(clamped[t, j]))
            ref += float(wts[t, j]) * y
        for sh in range(w.S):
            _, _, y = oracle.pair_output(od, tok.x_q, tok.x_scale, bank.w13, bank.s13, bank.w2, bank.s2, t, w.E + sh)
            ref += y
        rms = np.sqrt(np.mean(ref ** 2)) + 1e-30
        assert np.max(np.abs(out[t] - ref)) <= 2e-2 * rms, f"token {t}"

