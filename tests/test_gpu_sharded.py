"""A vocabulary split into shards on one GPU, run in lockstep by one process: every shard's one-step walk
(whead_walk_keys with its v_offset) gives its winning packed key, the keys are merged by their maximum, and
whead_advance moves the state to the merged winner. Each row's projection and the advance use the same
arithmetic as the unsharded walk, so tokens and states must equal it bit for bit (and match the oracle)."""
import numpy as np
import pytest

import whead_inputs as I
from oracle import oracle as O
from parity_helpers import GAP, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    from speculative_decoding_serial_gb300 import build
    build.build()
    return torch


CASES = [
    # kind, V, r, B, gamma, T, shards
    (O.MARKOV, 20011, 256, 2, 5, 0.0, 2),
    (O.MARKOV, 20011, 256, 1, 5, 1.0, 3),
    (O.RECURRENT, 9000, 128, 2, 4, 0.0, 2),
    (O.RECURRENT, 9000, 256, 1, 4, 0.7, 3),
    (O.MARKOV, 151936, 256, 1, 6, 0.0, 4),
]


@pytest.mark.parametrize("kind,V,r,B,gamma,T,nshards", CASES)
def test_sharded_walk_is_the_unsharded_walk(torch_cuda, kind, V, r, B, gamma, T, nshards):
    torch = torch_cuda
    from speculative_decoding_serial_gb300 import sharded as S
    from speculative_decoding_serial_gb300 import whead as wh
    d = I.make_inputs(kind, V, r, B, gamma, seed=V + nshards)
    dd = to_device(d, "cuda")
    seed = 5
    full = wh.Head(dd["W"], dd["E"], kind=kind, A=dd["A"], c=dd["c"], max_B=B, max_gamma=gamma)
    tok_full = torch.empty((B, gamma), dtype=torch.int32, device="cuda")
    st_full = torch.empty((B, gamma, r), dtype=torch.float32, device="cuda")
    full.walk_ex(dd["base"], dd["s0"], T=T, seed=seed, out_tokens=tok_full, out_state=st_full)
    assert full.status() == 0
    full.close()

    heads, bases = [], []
    for k in range(nshards):
        lo, hi = S.shard_bounds(V, nshards, k)
        heads.append(wh.Head(dd["W"][lo:hi].contiguous(), dd["E"], kind=kind, A=dd["A"], c=dd["c"], max_B=B,
                             max_gamma=1, v_offset=lo, e_rows=V))
        bases.append(dd["base"][:, :, lo:hi].contiguous())

    def step(t, s):
        keys = []
        for h, b in zip(heads, bases):
            _, k = h.walk_keys(b[:, t:t + 1].contiguous(), s.contiguous(), T=T, seed=seed, t0=t)
            keys.append(S.to_ordered(k[:, 0]))
        return S.from_ordered(torch.stack(keys).max(dim=0).values)

    def advance(x, s):
        nxt = torch.empty_like(s)
        return heads[0].advance(x.contiguous(), s.contiguous(), nxt)

    toks, states = S.ShardedWalk(step, lambda v: v, advance).walk(dd["s0"], gamma)
    for h in heads:
        assert h.status() == 0
        h.close()
    np.testing.assert_array_equal(toks.cpu().numpy(), tok_full.cpu().numpy())
    np.testing.assert_array_equal(states.cpu().numpy(), st_full.cpu().numpy())
    ref = O.walk(kind, d["W"], d["E"], d["base"], d["s0"], A=d["A"], c=d["c"], T=T, seed=seed)
    assert ((toks.cpu().numpy() == ref["tokens"]) | (ref["gap"] <= GAP)).all()


def test_shard_offset_must_be_group_aligned(torch_cuda):
    from speculative_decoding_serial_gb300 import whead as wh
    d = I.make_inputs(O.MARKOV, 1000, 64, 1, 2, seed=1)
    dd = to_device(d, "cuda")
    with pytest.raises(wh.WheadError) as e:
        wh.Head(dd["W"][8:].contiguous(), dd["E"], kind=O.MARKOV, v_offset=8, e_rows=1000)
    assert e.value.code == wh.ERR_INVALID_ARG
