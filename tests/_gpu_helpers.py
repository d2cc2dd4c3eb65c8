"""Shared pieces of the GPU parity tests: cached inputs and the tolerance check."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from bit_moe_expert_router_gb300 import binding, synth

# Output tolerance of the layer (relative to the oracle output's rms):
# max |err| <= 2e-2 * rms and at least 99.9% of elements within 1e-2 * rms.
MAX_REL = 2e-2
BULK_REL = 1e-2
BULK_FRAC = 0.999


@functools.lru_cache(maxsize=4)
def _bank_for(H, I, E, S, g, twobit_frac, seed):
    w = synth.Workload("bank", T=1, H=H, I=I, E=E, S=S, top_k=1, group=g, twobit_frac=twobit_frac, seed=seed)
    return synth.make_bank(w)


def bank_of(w: synth.Workload) -> synth.Bank:
    return _bank_for(w.H, w.I, w.E, w.S, w.group, w.twobit_frac, w.seed)


@functools.lru_cache(maxsize=4)
def _device_bank(H, I, E, S, g, twobit_frac, seed):
    b = _bank_for(H, I, E, S, g, twobit_frac, seed)
    dev = torch.device("cuda:0")
    return tuple(torch.from_numpy(a).to(dev) for a in (b.w13, b.s13, b.w2, b.s2))


def device_bank(w: synth.Workload):
    return _device_bank(w.H, w.I, w.E, w.S, w.group, w.twobit_frac, w.seed)


def dims(w: synth.Workload) -> binding.Dims:
    return binding.dims_of(w.T, w.H, w.I, w.E, w.S, w.top_k, w.group)


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")


def run_forward(w: synth.Workload, tok: synth.Tokens, bank_dev=None) -> np.ndarray:
    w13, s13, w2, s2 = bank_dev if bank_dev is not None else device_bank(w)
    d = dims(w)
    out = torch.full((w.T, w.H), float("nan"), dtype=torch.float32, device="cuda:0")
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    binding.moe_w4a8_forward(to_dev(tok.x_q), to_dev(tok.x_scale), to_dev(tok.logits), w13, s13, w2, s2, d, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    pick = rng.choice(np.arange(1, T - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, T - 1], pick]))


def assert_output_close(out: np.ndarray, ref: np.ndarray, what: str = ""):
    out = np.asarray(out, dtype=np.float64)
    assert out.shape == ref.shape
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = np.abs(out - ref)
    if rms == 0.0:
        assert float(err.max(initial=0.0)) == 0.0, f"{what}: reference is zero, output is not"
        return
    worst = float(err.max()) / rms
    bulk = float(np.mean(err <= BULK_REL * rms))
    assert worst <= MAX_REL, f"{what}: max|err|/rms = {worst:.3e} > {MAX_REL}"
    assert bulk >= BULK_FRAC, f"{what}: only {bulk:.5f} of elements within {BULK_REL} rms"


def oracle_out(w, tok, bank, tokens=None):
    return oracle.forward_workload(w, tok, bank, tokens)
