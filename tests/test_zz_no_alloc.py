"""The allocation-free walk (whead_walk_noalloc) against the regular entry point (whead_walk).

whead_walk_noalloc serves callers that may not allocate device memory themselves: engines that own all
GPU memory in their own pool, and loops that cannot take the device synchronization of cudaMalloc. Its
scratch is one fixed device array inside the library, shared by every call. This test calls it through
the C ABI twice in a row for each case (so the second call runs on the array the first call left behind)
and compares tokens and fp32 logits with whead_walk on the same inputs, under the parity tolerance used by
the other GPU tests (tokens identical; logits within 2e-2 times the logit RMS; here they are identical,
since both run the same kernel). Around the second call it also checks that the device's free memory does
not change. It lives in its own file so that pytest collects it last.
"""
import gc

import numpy as np
import pytest

import whead_inputs as I

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-2


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    from speculative_decoding_serial_gb300 import build
    build.build()
    return torch


@pytest.mark.parametrize("kind,V,r,B,gamma,T", [
    (0, 151936, 256, 1, 16, 0.0),   # full vocabulary, fully resident (shared + tensor memory + registers)
    (0, 9001, 128, 3, 5, 1.0),      # ragged vocabulary, sampled
    (1, 20000, 256, 2, 4, 0.0),     # recurrent head (uses the A h slices of the scratch)
])
def test_noalloc_matches_regular_entry_point_twice(torch_cuda, kind, V, r, B, gamma, T):
    torch = torch_cuda
    from speculative_decoding_serial_gb300 import whead as wh

    d = I.make_inputs(kind, V, r, B, gamma, seed=17)
    dev = "cuda"
    W = torch.from_numpy(d["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    E = torch.from_numpy(d["E"].view(np.int16)).view(torch.bfloat16).to(dev)
    base = torch.from_numpy(d["base"]).to(dev)
    s0 = torch.from_numpy(d["s0"]).to(dev)
    A = None if d["A"] is None else torch.from_numpy(d["A"]).to(dev)
    c = None if d["c"] is None else torch.from_numpy(d["c"]).to(dev)

    head = wh.Head(W, E, kind=kind, A=A, c=c, max_B=B, max_gamma=gamma, flags=wh.FLAG_LOGITS_F32)
    ref_tok = torch.empty((B, gamma), dtype=torch.int32, device=dev)
    ref_z = torch.empty((B, gamma, V), dtype=torch.float32, device=dev)
    head.walk(base, s0, T=T, seed=99, out_tokens=ref_tok, out_logits=ref_z)
    assert head.status() == 0
    ref_tok, ref_z = ref_tok.cpu().numpy(), ref_z.cpu().numpy()
    head.close()
    scale = float(np.sqrt(np.mean(ref_z.astype(np.float64) ** 2)))

    for call in range(2):
        tok = torch.full((B, gamma), -1, dtype=torch.int32, device=dev)
        z = torch.full((B, gamma, V), float("nan"), dtype=torch.float32, device=dev)
        status = torch.full((1,), 12345, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()
        # the first call on a device may load the library's device code (and with it the scratch array); the
        # second call must leave the device's free memory and torch's allocations exactly as they were (the
        # garbage collector is held off meanwhile, so that no unrelated tensor is freed during the call)
        gc.collect()
        gc.disable()
        try:
            free0, held0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
            wh.walk_noalloc(W, E, base, s0, kind=kind, A=A, c=c, T=T, seed=99, flags=wh.FLAG_LOGITS_F32,
                            out_tokens=tok, out_logits=z, out_status=status)
            torch.cuda.synchronize()
            free1, held1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        finally:
            gc.enable()
        if call == 1:
            assert free1 == free0, "the call changed the device's free memory"
            assert held1 == held0, "the call allocated through torch"
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        np.testing.assert_array_equal(tok.cpu().numpy(), ref_tok, err_msg=f"call {call}")
        assert np.max(np.abs(z.cpu().numpy() - ref_z)) <= LOGIT_TOL * scale, f"call {call}"


def test_noalloc_rejects_sizes_beyond_its_scratch(torch_cuda):
    torch = torch_cuda
    from speculative_decoding_serial_gb300 import whead as wh

    d = I.make_inputs(0, 1000, 64, 1, 2, seed=1)
    W = torch.from_numpy(d["W"].view(np.int16)).view(torch.bfloat16).cuda()
    E = torch.from_numpy(d["E"].view(np.int16)).view(torch.bfloat16).cuda()
    base = torch.zeros((17, 2, 1000), dtype=torch.float32, device="cuda")   # 17 walks > 16
    s0 = torch.zeros((17, 64), dtype=torch.float32, device="cuda")
    tok = torch.empty((17, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(wh.WheadError) as e:
        wh.walk_noalloc(W, E, base, s0, out_tokens=tok)
    assert e.value.code == wh.ERR_UNSUPPORTED


def test_noalloc_reports_a_timeout_and_the_next_call_is_correct(torch_cuda):
    """A walk whose bounded waits run out (CTA 0 skips its first arrival: a host flag, no fault) reports
    WHEAD_ERR_TIMEOUT through the caller's status word (and check=True raises it); the next call on the same shared
    scratch array, which the call clears first, gives the regular entry point's tokens again."""
    torch = torch_cuda
    from speculative_decoding_serial_gb300 import whead as wh

    d = I.make_inputs(0, 40000, 128, 2, 3, seed=2)
    W = torch.from_numpy(d["W"].view(np.int16)).view(torch.bfloat16).cuda()
    E = torch.from_numpy(d["E"].view(np.int16)).view(torch.bfloat16).cuda()
    base = torch.from_numpy(d["base"]).cuda()
    s0 = torch.from_numpy(d["s0"]).cuda()
    tok = torch.empty((2, 3), dtype=torch.int32, device="cuda")
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    with pytest.raises(wh.WheadError) as e:
        wh.walk_noalloc(W, E, base, s0, flags=wh.FLAG_FAULT_SKIP_ARRIVAL, timeout_us=20000, out_tokens=tok,
                        out_status=status, check=True)
    assert e.value.code == wh.ERR_TIMEOUT
    assert int(status.item()) == wh.ERR_TIMEOUT
    head = wh.Head(W, E, kind=0, max_B=2, max_gamma=3)
    ref = head.walk(base, s0).cpu().numpy()
    assert head.status() == 0
    head.close()
    wh.walk_noalloc(W, E, base, s0, out_tokens=tok, out_status=status, check=True)
    np.testing.assert_array_equal(tok.cpu().numpy(), ref)
