"""GPU parity at the edges of what the boundary accepts ("Weights That Stay", Fig. 2's walk and Fig. 8's selection
at degenerate and maximal shapes): vocabularies of one row and of less than one 16-row group, ragged batches at
the longest walk (64 steps), 16 walks at the longest walk on the full 151,936-row vocabulary, and the largest
vocabulary the placement accepts on this GPU (255 groups of 16 rows per CTA), with the next row rejected.
The oracle splits each step's rows over the host's cores here (its results do not depend on the thread count).
"""
import os

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
    O.set_threads(os.cpu_count() or 1)
    yield torch
    O.set_threads(1)


def head_for(d, dd, B, gamma, flags=0):
    from speculative_decoding_serial_gb300 import whead as wh
    return wh.Head(dd["W"], dd["E"], kind=d["kind"], A=dd["A"], c=dd["c"], max_B=B, max_gamma=gamma,
                   flags=flags | wh.FLAG_LOGITS_F32)


@pytest.mark.parametrize("V", [1, 2, 15, 16, 17])
@pytest.mark.parametrize("B,T", [(1, 0.0), (3, 1.0)])
def test_tiny_vocabularies(torch_cuda, V, B, T):
    """Less than one 16-row group (one CTA, rows past V zero-filled and never selected); V = 1 has one token."""
    d = I.make_inputs(O.MARKOV, V, 64, B, 4, seed=100 + V)
    dd = to_device(d, "cuda")
    head = head_for(d, dd, B, 4)
    ref, _ = check_walk(head, d, dd, T=T, seed=3)
    if V == 1:
        assert (ref["tokens"] == 0).all()
    head.close()


@pytest.mark.parametrize("kind,V,r,B", [(O.MARKOV, 20011, 192, 9), (O.RECURRENT, 9001, 128, 3)])
def test_longest_walk_ragged_batch(torch_cuda, kind, V, r, B):
    """64 steps (the most a handle accepts), a rank of three 64-wide boxes and a second, partial batch half."""
    d = I.make_inputs(kind, V, r, B, 64, seed=V + B)
    dd = to_device(d, "cuda")
    head = head_for(d, dd, B, 64)
    near = []
    check_walk(head, d, dd, T=1.0, seed=21, report=near)
    print("near-tie steps:", near)
    head.close()


@pytest.mark.parametrize("B,gamma", [(16, 64), (1, 64)])
def test_full_vocabulary_largest_batch_and_walk(torch_cuda, B, gamma):
    """V = 151,936, r = 256 at the largest batch and the longest walk, through the call the benchmark times (no
    logits): partially resident at 16 walks, fully resident at one."""
    d = I.make_inputs(O.MARKOV, 151936, 256, B, gamma, seed=7)
    dd = to_device(d, "cuda")
    from speculative_decoding_serial_gb300 import whead as wh
    head = wh.Head(dd["W"], dd["E"], kind=O.MARKOV, max_B=B, max_gamma=gamma)
    near = []
    check_walk(head, d, dd, T=0.0, seed=0, want_z=False, report=near)
    print(head.plan(B), "near-tie steps:", near)
    head.close()


def test_largest_vocabulary_the_placement_accepts(torch_cuda):
    """255 groups of 16 rows per CTA on every SM (up to 256 CTAs) is the most a walk can place; one row more is
    rejected with WHEAD_ERR_UNSUPPORTED, and the largest is walked at parity (mostly on chip, the rest streamed)."""
    torch = torch_cuda
    from speculative_decoding_serial_gb300 import whead as wh
    sms = min(torch.cuda.get_device_properties(0).multi_processor_count, 256)
    V = 255 * 16 * sms
    W1 = torch.zeros((V + 1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(wh.WheadError) as e:
        wh.Head(W1, W1, kind=O.MARKOV, max_B=1, max_gamma=2)
    assert e.value.code == wh.ERR_UNSUPPORTED
    del W1
    d = I.make_inputs(O.MARKOV, V, 64, 1, 2, seed=5)
    dd = to_device(d, "cuda")
    head = head_for(d, dd, 1, 2)
    plan = head.plan(1)
    assert plan["groups_per_cta"] == 255, plan
    print(plan)
    check_walk(head, d, dd, T=1.0, seed=9)
    head.close()
