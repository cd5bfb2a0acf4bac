"""GPU parity of the E4M3-weight walk (the pages' Fig. 7 two-vector projection with the 8-bit float format):
the device quantizer against the oracle's bit for bit, and the walk against the oracle's E4M3 walk on the
same seeded inputs, with the tolerances of the bf16 path."""
import ctypes

import numpy as np
import pytest

import whead_inputs as I
from oracle import oracle as O
from parity_helpers import check_walk, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    from speculative_decoding_serial_gb300 import build
    build.build()
    return torch


@pytest.mark.parametrize("V,r", [(1, 128), (37, 128), (1000, 256), (20011, 256)])
def test_device_quantizer_matches_oracle(torch_cuda, V, r):
    torch = torch_cuda
    from speculative_decoding_serial_gb300 import whead as wh
    d = I.make_inputs(O.MARKOV, V, r, 1, 1, seed=V)
    W = d["W"].copy()
    W[0, :] = 0  # an all-zero row: scale 0, zero codes
    Wd = torch.from_numpy(W.view(np.int16)).view(torch.bfloat16).cuda()
    Wq = torch.empty((V, r), dtype=torch.uint8, device="cuda")
    sw = torch.empty(V, dtype=torch.float32, device="cuda")
    rc = wh.load().whead_quantize_w_e4m3(ctypes.c_void_p(Wd.data_ptr()), V, r, ctypes.c_void_p(Wq.data_ptr()),
                                        ctypes.c_void_p(sw.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    want_q, want_s = O.quantize_w_e4m3(W)
    np.testing.assert_array_equal(Wq.cpu().numpy(), want_q)
    np.testing.assert_array_equal(sw.cpu().numpy(), want_s)


E4M3_CASES = [
    # kind, V, r, B, gamma, T, grid
    (O.MARKOV, 1000, 128, 1, 4, 0.0, 0),
    (O.MARKOV, 4097, 256, 1, 5, 0.0, 0),
    (O.MARKOV, 5003, 256, 2, 4, 0.0, 7),
    (O.MARKOV, 20011, 256, 4, 5, 0.0, 0),
    (O.MARKOV, 9000, 128, 3, 4, 1.0, 0),
    (O.MARKOV, 20011, 256, 1, 6, 0.7, 0),
    (O.RECURRENT, 3001, 128, 1, 5, 0.0, 0),
    (O.RECURRENT, 9000, 256, 2, 4, 0.0, 0),
    (O.MARKOV, 30000, 128, 2, 4, 0.0, 152),
]


@pytest.mark.parametrize("kind,V,r,B,gamma,T,grid", E4M3_CASES)
def test_e4m3_small_parity(torch_cuda, kind, V, r, B, gamma, T, grid):
    from speculative_decoding_serial_gb300 import whead as wh
    d = I.make_inputs(kind, V, r, B, gamma, seed=V + r + B + 7)
    dd = to_device(d, "cuda")
    head = wh.Head(dd["W"], dd["E"], kind=kind, A=dd["A"], c=dd["c"], max_B=B, max_gamma=gamma, grid=grid,
                   flags=wh.FLAG_W_E4M3 | wh.FLAG_LOGITS_F32)
    near = []
    check_walk(head, d, dd, T=T, seed=99, report=near, w_e4m3=O.quantize_w_e4m3(d["W"]))
    if near:
        print("near-tie steps:", near)
    head.close()


@pytest.mark.parametrize("name", ["markov_v151936_r256_b1_g16_e4m3", "markov_v248064_r256_b1_g16_e4m3",
                                  "markov_v248064_r256_b4_g16_e4m3"])
def test_e4m3_workload_parity(torch_cuda, name):
    from speculative_decoding_serial_gb300 import whead as wh
    w = I.WORKLOADS[name]
    d = I.workload_inputs(name)
    dd = to_device(d, "cuda")
    head = wh.Head(dd["W"], dd["E"], kind=w["kind"], max_B=w["B"], max_gamma=w["gamma"],
                   flags=wh.FLAG_W_E4M3 | wh.FLAG_LOGITS_F32)
    plan = head.plan(w["B"])
    print(name, plan)
    assert plan["stream_groups"] == 0  # E4M3 weights keep even the 248k vocabulary on chip
    near = []
    check_walk(head, d, dd, T=w["T"], seed=0, report=near, w_e4m3=O.quantize_w_e4m3(d["W"]))
    print("near-tie steps:", near)
    head.close()


def test_e4m3_rejects_unsupported_shapes(torch_cuda):
    from speculative_decoding_serial_gb300 import whead as wh
    d = I.make_inputs(O.MARKOV, 1000, 64, 1, 2, seed=1)
    dd = to_device(d, "cuda")
    with pytest.raises(wh.WheadError) as e:
        wh.Head(dd["W"], dd["E"], kind=O.MARKOV, flags=wh.FLAG_W_E4M3)  # r = 64
    assert e.value.code == wh.ERR_UNSUPPORTED
    d = I.make_inputs(O.MARKOV, 1000, 128, 1, 2, seed=1)
    dd = to_device(d, "cuda")
    with pytest.raises(wh.WheadError) as e:
        wh.Head(dd["W"], dd["E"], kind=O.MARKOV, max_B=5, flags=wh.FLAG_W_E4M3)  # more than 4 walks
    assert e.value.code == wh.ERR_UNSUPPORTED
