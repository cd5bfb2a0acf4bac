"""GPU parity: the CUDA walk (through the C ABI) against the CPU oracle on the same seeded inputs.

Covers the Fig. 2 walk structure ("Weights That Stay", Fig. 2), the single rounding of base-added
logits (Fig. 7), the cross-CTA selection (Fig. 8), Markov and recurrent heads (abstract), sampling at
T > 0, ragged vocabularies, several ranks and batch sizes, resume from any step, determinism, the
host-buffer entry point and the bounded-wait failure path.
"""
import numpy as np
import pytest

import whead_inputs as I
from oracle import oracle as O
from parity_helpers import GAP, LOGIT_TOL, bf16_to_f32, check_walk, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    from speculative_decoding_serial_gb300 import build
    build.build()
    return torch


def make_head(torch_cuda, d, dd, *, max_B, max_gamma, flags=0, grid=0, timeout_us=0):
    from speculative_decoding_serial_gb300 import whead as wh
    return wh.Head(dd["W"], dd["E"], kind=d["kind"], A=dd["A"], c=dd["c"], max_B=max_B, max_gamma=max_gamma,
                   flags=flags | wh.FLAG_LOGITS_F32, grid=grid, timeout_us=timeout_us)


SMALL = [
    # kind, V, r, B, gamma, T, grid
    (O.MARKOV, 12 * 16, 64, 1, 3, 0.0, 0),
    (O.MARKOV, 1000, 64, 1, 4, 0.0, 0),
    (O.MARKOV, 4097, 128, 3, 5, 0.0, 0),
    (O.MARKOV, 5003, 192, 2, 4, 0.0, 7),
    (O.MARKOV, 20011, 256, 1, 6, 0.0, 0),
    (O.MARKOV, 20011, 256, 8, 3, 0.0, 0),
    (O.MARKOV, 7777, 256, 9, 3, 0.0, 0),
    (O.MARKOV, 7777, 128, 16, 2, 0.0, 0),
    (O.MARKOV, 3001, 64, 4, 5, 1.0, 0),
    (O.MARKOV, 9000, 256, 2, 4, 0.7, 0),
    # one sampled walk (the single-walk selection scan draws four rows' noise per Philox call)
    (O.MARKOV, 5003, 128, 1, 5, 1.0, 0),
    (O.MARKOV, 20011, 256, 1, 6, 0.7, 0),
    (O.MARKOV, 30000, 64, 1, 4, 1.0, 152),
    (O.RECURRENT, 3001, 64, 1, 4, 1.0, 0),
    (O.RECURRENT, 3001, 64, 1, 5, 0.0, 0),
    (O.RECURRENT, 9000, 256, 2, 4, 0.0, 0),
    (O.RECURRENT, 4000, 128, 3, 4, 1.0, 0),
    # many CTAs with few groups each: every CTA takes part in the exchange
    (O.MARKOV, 30000, 64, 2, 4, 0.0, 152),
]


@pytest.mark.parametrize("kind,V,r,B,gamma,T,grid", SMALL)
def test_small_parity(torch_cuda, kind, V, r, B, gamma, T, grid):
    d = I.make_inputs(kind, V, r, B, gamma, seed=V + r + B)
    dd = to_device(d, "cuda")
    head = make_head(torch_cuda, d, dd, max_B=B, max_gamma=gamma, grid=grid)
    near = []
    check_walk(head, d, dd, T=T, seed=1234, report=near)
    if near:
        print("near-tie steps:", near)
    head.close()


def test_bf16_logits_single_rounding(torch_cuda):
    """Fig. 7: the projection is added to the base logits and rounded once. The bf16 logits of a walk must be
    the round-to-nearest-even bf16 of the same walk's fp32 z, bit for bit; and against the oracle's bf16(z)
    they may differ only by one bf16 ulp, and only where the oracle's z lies within |z_gpu - z_oracle| of the
    rounding midpoint between the two values (the logits rule of the parity tolerances). Tokens follow the
    per-step gap rule: logits are compared up to the first step where a walk diverged at a near tie."""
    from speculative_decoding_serial_gb300 import whead as wh
    torch = torch_cuda
    B, gamma, V = 2, 3, 6000
    d = I.make_inputs(O.MARKOV, V, 128, B, gamma, seed=5)
    dd = to_device(d, "cuda")
    head = wh.Head(dd["W"], dd["E"], kind=O.MARKOV, max_B=B, max_gamma=gamma)
    lg = torch.empty((B, gamma, V), dtype=torch.bfloat16, device="cuda")
    tok = head.walk(dd["base"], dd["s0"], out_logits=lg).cpu().numpy()
    assert head.status() == 0
    head.close()
    head32 = make_head(torch_cuda, d, dd, max_B=B, max_gamma=gamma)  # same walk, fp32 z emitted
    z32 = torch.empty((B, gamma, V), dtype=torch.float32, device="cuda")
    tok32 = head32.walk(dd["base"], dd["s0"], out_logits=z32).cpu().numpy()
    assert head32.status() == 0
    head32.close()
    np.testing.assert_array_equal(tok, tok32)
    got_bits = lg.view(torch.int16).cpu().numpy().view(np.uint16)
    z32 = z32.cpu().numpy()
    # (1) single rounding: the emitted bf16 is RNE(z) of the walk's own fp32 z
    np.testing.assert_array_equal(got_bits, I.to_bf16_bits(z32))
    # (2) against the oracle, step by step up to the first near-tie divergence
    ref = O.walk(O.MARKOV, d["W"], d["E"], d["base"], d["s0"], want_z=True, want_logits=True)
    last = gamma
    for t in range(gamma):
        bad = [b for b in range(B) if tok[b, t] != ref["tokens"][b, t]]
        for b in bad:
            assert ref["gap"][b, t] <= GAP, f"walk {b} step {t}: token mismatch with gap {ref['gap'][b, t]}"
        if bad:
            last = t + 1  # this step's logits used the same state on both sides; later steps may not
            break
    got = bf16_to_f32(got_bits[:, :last])
    want = bf16_to_f32(ref["logits"][:, :last])
    zg, zo = z32[:, :last].astype(np.float64), ref["z"][:, :last].astype(np.float64)
    diff = got != want
    if diff.any():
        def ordered(bits):  # bf16 bit patterns to integers in the order of their values
            b = np.asarray(bits).astype(np.int64)
            return np.where(b & 0x8000, 0xFFFF - b, b | 0x8000)
        steps = np.abs(ordered(got_bits[:, :last]) - ordered(ref["logits"][:, :last]))[diff]
        assert np.all(steps == 1), "bf16 logits differ by more than one bf16 ulp"
        lo, hi = np.minimum(got, want)[diff].astype(np.float64), np.maximum(got, want)[diff].astype(np.float64)
        mid = (lo + hi) / 2.0
        assert np.all(np.abs(zo[diff] - mid) <= np.abs(zg[diff] - zo[diff])), \
            "a bf16 mismatch away from a rounding midpoint"
    print(f"bf16 logits: {int(diff.sum())} of {diff.size} differ from the oracle's, each at a rounding midpoint")


@pytest.mark.parametrize("kind,B", [(O.RECURRENT, 2), (O.MARKOV, 1)])
def test_resume_from_any_step_bit_exact(torch_cuda, kind, B):
    torch = torch_cuda
    d = I.make_inputs(kind, 8000, 128, B, 6, seed=9)
    dd = to_device(d, "cuda")
    head = make_head(torch_cuda, d, dd, max_B=B, max_gamma=6)
    full = run_gpu(head, dd, B, 6, 1.0, 77)
    for t0 in range(1, 6):
        part = run_gpu(head, dd, B, 6 - t0, 1.0, 77, t0=t0, base=dd["base"][:, t0:].contiguous(),
                       s0=torch.from_numpy(full["state"][:, t0 - 1].copy()).cuda())
        np.testing.assert_array_equal(part["tokens"], full["tokens"][:, t0:])
        np.testing.assert_array_equal(part["z"], full["z"][:, t0:])
        np.testing.assert_array_equal(part["state"], full["state"][:, t0:])
    head.close()


def test_deterministic(torch_cuda):
    d = I.make_inputs(O.MARKOV, 50000, 256, 4, 5, seed=3)
    dd = to_device(d, "cuda")
    head = make_head(torch_cuda, d, dd, max_B=4, max_gamma=5)
    a = run_gpu(head, dd, 4, 5, 1.0, 5)
    b = run_gpu(head, dd, 4, 5, 1.0, 5)
    for k in ("tokens", "z", "state"):
        np.testing.assert_array_equal(a[k], b[k])
    head.close()


def test_host_entry_point_matches_device(torch_cuda):
    from speculative_decoding_serial_gb300 import whead as wh
    torch = torch_cuda
    d = I.make_inputs(O.MARKOV, 10000, 128, 2, 4, seed=21)
    dd = to_device(d, "cuda")
    head = wh.Head(dd["W"], dd["E"], kind=O.MARKOV, max_B=2, max_gamma=4)
    dev_tok = head.walk(dd["base"], dd["s0"], T=1.0, seed=8).cpu()
    base_h = torch.from_numpy(d["base"]).pin_memory()
    s0_h = torch.from_numpy(d["s0"]).pin_memory()
    host_tok = head.walk_host(base_h, s0_h, T=1.0, seed=8)
    assert torch.equal(dev_tok, host_tok)
    head.close()


@pytest.mark.parametrize("memory", ["pinned", "pageable", "staged", "u0_unaligned"])
def test_host_entry_point_base_in_place_or_staged(torch_cuda, memory):
    """whead_walk_host reads the base logits and u0, and writes the tokens, where they lie when the GPU can
    address them (pinned memory; any host memory where the GPU walks the host's page tables), and copies them
    otherwise or when asked to (FLAG_HOST_STAGE; a u0 off a 16-byte boundary is copied too); tokens and logits
    must equal those of the walk on device buffers, call after call."""
    from speculative_decoding_serial_gb300 import whead as wh
    torch = torch_cuda
    d = I.make_inputs(O.MARKOV, 20011, 256, 3, 16, seed=33)
    dd = to_device(d, "cuda")
    flags = wh.FLAG_LOGITS_F32 | (wh.FLAG_HOST_STAGE if memory == "staged" else 0)
    head = wh.Head(dd["W"], dd["E"], kind=O.MARKOV, max_B=3, max_gamma=16, flags=flags)
    lg_dev = torch.empty((3, 16, 20011), dtype=torch.float32, device="cuda")
    dev_tok = head.walk(dd["base"], dd["s0"], T=1.0, seed=4, out_logits=lg_dev).cpu()
    base_h = torch.from_numpy(d["base"])
    s0_h = torch.from_numpy(d["s0"])
    lg_host = torch.empty((3, 16, 20011), dtype=torch.float32)
    if memory == "pinned":
        base_h, s0_h, lg_host = base_h.pin_memory(), s0_h.pin_memory(), lg_host.pin_memory()
    if memory == "u0_unaligned":
        buf = torch.empty(s0_h.numel() + 1, dtype=torch.float32)
        s0_h = buf[1:].view(s0_h.shape)  # 4 bytes past an allocation's start
        s0_h.copy_(torch.from_numpy(d["s0"]))
        assert s0_h.data_ptr() % 16 != 0
    for k in range(3):
        if k == 2:
            base_h = base_h.clone()  # a different buffer on the last call
            base_h = base_h.pin_memory() if memory == "pinned" else base_h
        host_tok = head.walk_host(base_h, s0_h, T=1.0, seed=4, out_logits=lg_host)
        assert torch.equal(dev_tok, host_tok)
        assert torch.equal(lg_dev.cpu(), lg_host)
    assert head.status() == 0
    head.close()


HOST_VARIANTS = [
    # kind, V, r, B, gamma, T, flags: each kernel family of the host-buffer walk (asynchronous base copies
    # where the second buffer fits; at B = 16 it does not, and the walk reads host memory in place)
    (O.MARKOV, 30011, 256, 1, 6, 0.0, 0),
    (O.MARKOV, 30011, 256, 1, 6, 1.0, 0),
    (O.MARKOV, 12000, 64, 16, 3, 1.0, 0),
    (O.RECURRENT, 9001, 128, 1, 5, 0.0, 0),
    (O.RECURRENT, 9001, 192, 3, 4, 1.0, 0),
    (O.MARKOV, 20000, 256, 1, 5, 0.0, "e4m3"),
    (O.MARKOV, 20000, 128, 4, 4, 1.0, "e4m3"),
]


@pytest.mark.parametrize("kind,V,r,B,gamma,T,wfmt", HOST_VARIANTS)
def test_host_entry_point_kernel_variants(torch_cuda, kind, V, r, B, gamma, T, wfmt):
    """Tokens, logits and the device status of whead_walk_host on pinned host buffers equal those of the walk
    on device buffers with the same handle (bit for bit: the same arithmetic, another copy of the base logits)."""
    from speculative_decoding_serial_gb300 import whead as wh
    torch = torch_cuda
    d = I.make_inputs(kind, V, r, B, gamma, seed=V + B)
    dd = to_device(d, "cuda")
    flags = wh.FLAG_LOGITS_F32 | (wh.FLAG_W_E4M3 if wfmt == "e4m3" else 0)
    head = wh.Head(dd["W"], dd["E"], kind=kind, A=dd["A"], c=dd["c"], max_B=B, max_gamma=gamma, flags=flags)
    lg_dev = torch.empty((B, gamma, V), dtype=torch.float32, device="cuda")
    dev_tok = head.walk(dd["base"], dd["s0"], T=T, seed=11, out_logits=lg_dev).cpu()
    lg_host = torch.empty((B, gamma, V), dtype=torch.float32).pin_memory()
    host_tok = head.walk_host(torch.from_numpy(d["base"]).pin_memory(), torch.from_numpy(d["s0"]).pin_memory(),
                              T=T, seed=11, out_tokens=torch.empty((B, gamma), dtype=torch.int32).pin_memory(),
                              out_logits=lg_host)
    assert torch.equal(dev_tok, host_tok)
    assert torch.equal(lg_dev.cpu(), lg_host)
    assert head.status() == 0
    head.close()


def test_host_entry_point_reports_device_errors(torch_cuda):
    """A walk whose bounded waits run out makes whead_walk_host return WHEAD_ERR_TIMEOUT (and clear it)."""
    from speculative_decoding_serial_gb300 import whead as wh
    torch = torch_cuda
    d = I.make_inputs(O.MARKOV, 40000, 128, 1, 3, seed=2)
    dd = to_device(d, "cuda")
    bad = wh.Head(dd["W"], dd["E"], kind=O.MARKOV, max_B=1, max_gamma=3, flags=wh.FLAG_FAULT_SKIP_ARRIVAL,
                  timeout_us=20000)
    with pytest.raises(wh.WheadError) as err:
        bad.walk_host(torch.from_numpy(d["base"]), torch.from_numpy(d["s0"]))
    assert err.value.code == wh.ERR_TIMEOUT
    assert bad.status() == 0
    bad.close()


@pytest.mark.parametrize("B", [1, 4, 12])
def test_wait_limit_reports_timeout_and_context_survives(torch_cuda, B):
    """CTA 0 skips its first arrival (a host flag); every other CTA's bounded wait must run out. One walk waits in
    the exchange warp alone; several walks also wait in the warps that read each walk's slots."""
    from speculative_decoding_serial_gb300 import whead as wh
    d = I.make_inputs(O.MARKOV, 40000, 128, B, 3, seed=2)
    dd = to_device(d, "cuda")
    bad = wh.Head(dd["W"], dd["E"], kind=O.MARKOV, max_B=B, max_gamma=3, flags=wh.FLAG_FAULT_SKIP_ARRIVAL,
                  timeout_us=20000)
    bad.walk(dd["base"], dd["s0"])
    assert bad.status() == wh.ERR_TIMEOUT
    assert bad.status() == 0  # cleared after reading
    bad.close()
    good = wh.Head(dd["W"], dd["E"], kind=O.MARKOV, max_B=B, max_gamma=3)
    tok = good.walk(dd["base"], dd["s0"]).cpu().numpy()
    assert good.status() == 0
    ref = O.walk(O.MARKOV, d["W"], d["E"], d["base"], d["s0"])
    assert ((tok == ref["tokens"]) | (ref["gap"] <= GAP)).all()
    good.close()


def test_invalid_arguments(torch_cuda):
    from speculative_decoding_serial_gb300 import whead as wh
    torch = torch_cuda
    d = I.make_inputs(O.MARKOV, 1000, 64, 1, 2, seed=1)
    dd = to_device(d, "cuda")
    head = wh.Head(dd["W"], dd["E"], kind=O.MARKOV, max_B=1, max_gamma=2)
    big = torch.zeros((2, 2, 1000), dtype=torch.float32, device="cuda")
    with pytest.raises(wh.WheadError) as e:
        head.walk(big, torch.zeros((2, 64), device="cuda"))
    assert e.value.code == wh.ERR_INVALID_ARG
    with pytest.raises(wh.WheadError):
        head.walk(dd["base"], dd["s0"], T=-1.0)
    head.close()
    Wbad = torch.zeros((100, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(wh.WheadError) as e:
        wh.Head(Wbad, Wbad, kind=O.MARKOV)
    assert e.value.code == wh.ERR_UNSUPPORTED


# --- the workloads of the pages at full size -------------------------------------------------------
@pytest.mark.parametrize("name", ["markov_v4096_r64_b1_g4", "markov_v151936_r256_b1_g16",
                                  "recurrent_v151936_r256_b1_g15"])
def test_workload_parity(torch_cuda, name):
    w = I.WORKLOADS[name]
    d = I.workload_inputs(name)
    dd = to_device(d, "cuda")
    head = make_head(torch_cuda, d, dd, max_B=w["B"], max_gamma=w["gamma"])
    plan = head.plan(w["B"])
    print(name, plan)
    near = []
    check_walk(head, d, dd, T=w["T"], seed=0, report=near)
    print("near-tie steps:", near)
    head.close()


@pytest.mark.parametrize("B,T", [(1, 1.0), (2, 0.0), (4, 1.0), (8, 0.0)])
def test_sweep_points_full_vocab(torch_cuda, B, T):
    """Points of the batch x temperature sweep at V = 151,936, r = 256 (gamma 7)."""
    d = I.make_inputs(O.MARKOV, 151936, 256, B, 7, seed=0)
    dd = to_device(d, "cuda")
    head = make_head(torch_cuda, d, dd, max_B=B, max_gamma=7)
    assert head.plan(B)["stream_groups"] == 0
    check_walk(head, d, dd, T=T, seed=11)
    head.close()


def test_phase_trace_stamps_are_ordered(torch_cuda):
    torch = torch_cuda
    d = I.make_inputs(O.MARKOV, 60000, 256, 1, 4, seed=4)
    dd = to_device(d, "cuda")
    head = make_head(torch_cuda, d, dd, max_B=1, max_gamma=4)
    G = head.plan(1)["grid"]
    S = 4 + 8 * 4
    buf = torch.zeros((G, S), dtype=torch.int64, device="cuda")
    head.set_trace(buf)
    run_gpu(head, dd, 1, 4, 0.0, 0)
    a = buf.cpu().numpy()
    head.set_trace(None)
    clk = a[:, :S // 2]
    assert (clk > 0).all()
    assert (np.diff(clk, axis=1) >= 0).all()      # stamps of every CTA are in program order
    head.close()


# --- partial residency: groups that do not fit on chip are re-read from L2 every step -------------
STREAMED = [
    # kind, V, r, B, gamma, T, grid (a small grid forces most groups to stream)
    (O.MARKOV, 40000, 256, 1, 4, 0.0, 12),
    (O.MARKOV, 30011, 128, 3, 3, 1.0, 8),
    (O.RECURRENT, 20000, 256, 2, 3, 0.0, 6),
    (O.MARKOV, 40000, 256, 12, 2, 0.0, 24),
]


@pytest.mark.parametrize("kind,V,r,B,gamma,T,grid", STREAMED)
def test_streamed_parity(torch_cuda, kind, V, r, B, gamma, T, grid):
    d = I.make_inputs(kind, V, r, B, gamma, seed=V + B)
    dd = to_device(d, "cuda")
    head = make_head(torch_cuda, d, dd, max_B=B, max_gamma=gamma, grid=grid)
    plan = head.plan(B)
    assert plan["stream_groups"] > 0, plan
    check_walk(head, d, dd, T=T, seed=77)
    head.close()


@pytest.mark.parametrize("name", ["markov_v248064_r256_b1_g16", "markov_v248064_r256_b4_g16"])
def test_workload_parity_partial_residency(torch_cuda, name):
    w = I.WORKLOADS[name]
    d = I.workload_inputs(name)
    dd = to_device(d, "cuda")
    head = make_head(torch_cuda, d, dd, max_B=w["B"], max_gamma=w["gamma"])
    plan = head.plan(w["B"])
    print(name, plan)
    assert plan["stream_groups"] > 0
    near = []
    check_walk(head, d, dd, T=w["T"], seed=0, report=near)
    print("near-tie steps:", near)
    head.close()


def test_sweep_point_sixteen_walks(torch_cuda):
    """B = 16 at V = 151,936 (gamma 7, sampled): two batch halves, partially resident."""
    d = I.make_inputs(O.MARKOV, 151936, 256, 16, 7, seed=0)
    dd = to_device(d, "cuda")
    head = make_head(torch_cuda, d, dd, max_B=16, max_gamma=7)
    print(head.plan(16))
    check_walk(head, d, dd, T=1.0, seed=11)
    head.close()


def test_force_stream_parity(torch_cuda):
    """The fused but non-resident walk (every row of W re-read each step) gives the same walk."""
    from speculative_decoding_serial_gb300 import whead as wh
    d = I.make_inputs(O.MARKOV, 50000, 256, 2, 4, seed=31)
    dd = to_device(d, "cuda")
    head = make_head(torch_cuda, d, dd, max_B=2, max_gamma=4, flags=wh.FLAG_FORCE_STREAM)
    plan = head.plan(2)
    assert plan["smem_groups"] == plan["tmem_groups"] == plan["rf_groups"] == 0 and plan["stream_groups"] > 0
    check_walk(head, d, dd, T=1.0, seed=3)
    head.close()


# --- caller-chosen placements (the Fig. 12 placement sweep): any split of a CTA's groups over shared memory,
# tensor memory and registers, the rest streamed, gives the oracle's walk -------------------------------
CAPPED = [
    # B, (shared, tensor, register) caps
    (1, (4, 4, 2)),
    (2, (4, 4, 2)),
    (1, (0, 13, 0)),
    (3, (0, 0, 3)),
    (1, (13, 0, 0)),
    (1, (0, 0, 0)),
    # the shard load's ring: twelve staged groups through one slot (register groups in the last rounds), eight
    # through two slots with two batch halves, and as many staged groups as slots
    (1, (1, 8, 4)),
    (9, (2, 8, 0)),
    (1, (4, 4, 0)),
]


@pytest.mark.parametrize("B,caps", CAPPED)
def test_capped_placement_parity(torch_cuda, B, caps):
    from speculative_decoding_serial_gb300 import whead as wh
    d = I.make_inputs(O.MARKOV, 30011, 256, B, 4, seed=31 + B)
    dd = to_device(d, "cuda")
    head = wh.Head(dd["W"], dd["E"], kind=O.MARKOV, max_B=B, max_gamma=4, flags=wh.FLAG_LOGITS_F32, caps=caps)
    plan = head.plan(B)
    assert plan["smem_groups"] <= caps[0] and plan["tmem_groups"] <= caps[1] and plan["rf_groups"] <= caps[2]
    assert (plan["smem_groups"] + plan["tmem_groups"] + plan["rf_groups"] + plan["stream_groups"]
            == plan["groups_per_cta"])
    check_walk(head, d, dd, T=0.0, seed=3)
    head.close()


def test_capped_placement_rejects_negative_caps(torch_cuda):
    from speculative_decoding_serial_gb300 import whead as wh
    d = I.make_inputs(O.MARKOV, 1000, 64, 1, 2, seed=1)
    dd = to_device(d, "cuda")
    with pytest.raises(wh.WheadError) as e:
        wh.Head(dd["W"], dd["E"], kind=O.MARKOV, caps=(-1, 0, 0))
    assert e.value.code == wh.ERR_INVALID_ARG
