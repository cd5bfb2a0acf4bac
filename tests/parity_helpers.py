"""Shared helpers for the GPU-vs-oracle parity tests.

Tolerances (fixed before any kernel ran): logits max|z_gpu - z_oracle| <= 2e-2 * RMS(z_oracle); tokens
identical at every step whose oracle top-2 key gap exceeds 1e-2 (smaller gaps are reported, and the GPU
walk is resumed from the oracle's state after a divergence so that every later step is still checked);
recurrent state within 1e-5 * max(1, |h|).
"""
from __future__ import annotations

import numpy as np

import whead_inputs as I
from oracle import oracle as O

LOGIT_TOL = 2e-2
GAP = 1e-2
STATE_TOL = 1e-5


def to_device(d, dev):
    import torch
    out = {
        "W": torch.from_numpy(d["W"].view(np.int16)).view(torch.bfloat16).to(dev),
        "E": torch.from_numpy(d["E"].view(np.int16)).view(torch.bfloat16).to(dev),
        "base": torch.from_numpy(d["base"]).to(dev),
        "s0": torch.from_numpy(d["s0"]).to(dev),
        "A": None if d["A"] is None else torch.from_numpy(d["A"]).to(dev),
        "c": None if d["c"] is None else torch.from_numpy(d["c"]).to(dev),
    }
    return out


def bf16_to_f32(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def run_gpu(head, dd, B, gamma, T, seed, *, t0=0, base=None, s0=None, want_z=True, want_state=True):
    import torch
    dev = dd["base"].device
    base = dd["base"] if base is None else base
    s0 = dd["s0"] if s0 is None else s0
    tok = torch.empty((B, gamma), dtype=torch.int32, device=dev)
    z = torch.empty((B, gamma, head.V), dtype=torch.float32, device=dev) if want_z else None
    st = torch.empty((B, gamma, head.r), dtype=torch.float32, device=dev) if want_state else None
    head.walk_ex(base, s0, T=T, seed=seed, t0=t0, out_tokens=tok, out_logits=z, out_state=st)
    status = head.status()
    assert status == 0, f"device status {status}"
    return {"tokens": tok.cpu().numpy(), "z": None if z is None else z.cpu().numpy(),
            "state": None if st is None else st.cpu().numpy()}


def check_walk(head, d, dd, *, T=0.0, seed=0, check_state=True, report=None, w_e4m3=None, want_z=True, ref=None):
    """Full parity check of one call against the oracle, with the resume rule at near-tie divergences.
    w_e4m3: (Wq, sw) from the oracle's quantizer when the head runs with E4M3 weights.
    want_z=False runs the walk without logits (out_logits = NULL): for greedy walks that is the selection
    loop that scores keys only, the one the benchmark times. ref: the oracle's walk of these inputs, if the
    caller already has it (tokens, gap, state; z too when want_z)."""
    import torch
    kind = d["kind"]
    B, gamma, V = d["base"].shape
    if ref is None:
        ref = O.walk(kind, d["W"], d["E"], d["base"], d["s0"], A=d["A"], c=d["c"], T=T, seed=seed,
                     want_z=want_z, want_state=True, want_gap=True, w_e4m3=w_e4m3)
    scale = float(np.sqrt(np.mean(ref["z"].astype(np.float64) ** 2))) if want_z else None
    near = []
    t_start = 0
    s0 = dd["s0"]
    while t_start < gamma:
        base_part = dd["base"][:, t_start:].contiguous()
        got = run_gpu(head, dd, B, gamma - t_start, T, seed, t0=t_start, base=base_part, s0=s0, want_z=want_z)
        diverged_at = None
        for t in range(t_start, gamma):
            tt = t - t_start
            if want_z:
                zerr = np.max(np.abs(got["z"][:, tt] - ref["z"][:, t]))
                assert zerr <= LOGIT_TOL * scale, f"step {t}: max|dz| = {zerr} > {LOGIT_TOL} * {scale}"
            for b in range(B):
                if got["tokens"][b, tt] != ref["tokens"][b, t]:
                    assert ref["gap"][b, t] <= GAP, (
                        f"walk {b} step {t}: token {got['tokens'][b, tt]} != oracle {ref['tokens'][b, t]} "
                        f"with gap {ref['gap'][b, t]}")
                    near.append((b, t, float(ref["gap"][b, t])))
                    diverged_at = t
            if diverged_at is not None:
                break
            if check_state and kind == O.RECURRENT:
                err = np.abs(got["state"][:, tt] - ref["state"][:, t])
                lim = STATE_TOL * np.maximum(1.0, np.abs(ref["state"][:, t]))
                assert np.all(err <= lim), f"step {t}: state error {err.max()}"
            if check_state and kind == O.MARKOV:
                np.testing.assert_array_equal(got["state"][:, tt], ref["state"][:, t])
        if diverged_at is None:
            break
        # resume from the oracle's state after the near-tie step
        t_start = diverged_at + 1
        s0 = torch.from_numpy(np.ascontiguousarray(ref["state"][:, diverged_at])).to(dd["base"].device)
    if report is not None:
        report.extend(near)
    return ref, near
