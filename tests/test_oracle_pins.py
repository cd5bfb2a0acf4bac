"""Pins for the CPU oracle: each test ties it to something other than itself.

The oracle follows "Weights That Stay: On-Chip Megakernels for Serial Heads in Speculative Decoding"
(abstract; Fig. 2 shape V=12, r=4, three steps; Fig. 7 add-then-round-once; Fig. 8 one winner over all
rows). The pins are: a hand-computed walk, reductions to library routines (numpy matmul/argmax/tanh,
torch bf16 conversion, triton's Philox), closed forms (Gumbel moments, exact uniforms), invariants
(resume from any step, batch independence, lowest-index ties) and the Gumbel-max sampling law.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle as O
import whead_inputs as I

MARKOV, RECURRENT = 0, 1


def bf16_bits(x):
    return I.to_bf16_bits(np.asarray(x, dtype=np.float32))


def bf16_vals(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def lib_bf16_round_f32(x):
    """bf16 rounding by torch (library), returned as float32 values."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


# ---------------------------------------------------------------------------------------------
# 1. Hand-computed greedy walk on the Fig. 2 shape (V=12, r=4, 3 steps). Integer data is exact in
#    bf16 and fp32, so every z below is exact; step 0 has a tie between rows 4 and 5.
# ---------------------------------------------------------------------------------------------
HAND_W = [[1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 1, 0], [0, 0, 0, 1], [1, 1, 0, 0], [0, 1, 1, 0],
          [0, 0, 1, 1], [1, 0, 0, 1], [-1, 0, 1, 0], [0, -1, 0, 1], [2, 0, 0, 0], [0, 0, 0, 2]]
HAND_E = [[0, 0, 0, 1], [0, 0, 1, 0], [0, 1, 0, 0], [1, 0, 0, 0], [0, 0, 1, 1], [1, 1, 0, 0],
          [0, 1, 0, 1], [1, 0, 1, 0], [2, 0, 0, 0], [0, 2, 0, 0], [0, 0, 2, 0], [0, 0, 0, 2]]


def hand_inputs():
    W = bf16_bits(HAND_W)
    E = bf16_bits(HAND_E)
    base = np.zeros((1, 3, 12), dtype=np.float32)
    base[0, 0, 5] = 1.0
    base[0, 1, 3] = -1.0
    base[0, 1, 6] = 1.0
    base[0, 2, 0] = 3.0
    s0 = np.array([[1, 2, 0, 0]], dtype=np.float32)
    return W, E, base, s0


def test_hand_walk_markov():
    W, E, base, s0 = hand_inputs()
    out = O.walk(MARKOV, W, E, base, s0, want_z=True, want_logits=True, want_state=True)
    # t=0: u=(1,2,0,0): p=[1,2,0,0,3,2,0,1,-1,-2,2,0], +base[5]=1 -> tie at rows 4 and 5 -> 4
    # t=1: u=E[4]=(0,0,1,1): p=[0,0,1,1,0,1,2,1,1,1,0,2], base[3]=-1, base[6]=+1 -> row 6
    # t=2: u=E[6]=(0,1,0,1): p=[0,1,0,1,1,1,1,1,0,0,0,2], base[0]=+3 -> row 0
    z_hand = np.array([[1, 2, 0, 0, 3, 3, 0, 1, -1, -2, 2, 0],
                       [0, 0, 1, 0, 0, 1, 3, 1, 1, 1, 0, 2],
                       [3, 1, 0, 1, 1, 1, 1, 1, 0, 0, 0, 2]], dtype=np.float32)
    assert out["tokens"].tolist() == [[4, 6, 0]]
    np.testing.assert_array_equal(out["z"][0], z_hand)
    np.testing.assert_array_equal(bf16_vals(out["logits"][0]), z_hand)
    np.testing.assert_array_equal(out["gap"][0], [0.0, 1.0, 1.0])
    np.testing.assert_array_equal(out["state"][0], np.array([HAND_E[4], HAND_E[6], HAND_E[0]], np.float32))


def test_hand_walk_recurrent_zero_weights():
    # A = 0, c = 0: h1 = tanh(E[x0]); the projection then sees bf16(tanh(.)) values.
    W, E, base, s0 = hand_inputs()
    A = np.zeros((4, 4), np.float32)
    out = O.walk(RECURRENT, W, E, base, s0, A=A, c=np.zeros(4, np.float32), want_z=True, want_state=True)
    assert out["tokens"][0, 0] == 4                     # same first step as the Markov head
    h1 = np.tanh(np.array(HAND_E[4], np.float64)).astype(np.float32)
    np.testing.assert_array_equal(out["state"][0, 0], h1)
    q1 = lib_bf16_round_f32(h1).astype(np.float64)
    z1 = (np.array(HAND_W, np.float64) @ q1).astype(np.float32) + base[0, 1]
    np.testing.assert_array_equal(out["z"][0, 1], z1)
    assert out["tokens"][0, 1] == int(np.argmax(z1))


# ---------------------------------------------------------------------------------------------
# 2. Brute force on tiny random walks: re-derive every step with library routines.
# ---------------------------------------------------------------------------------------------
def rederive_markov(W, E, base, s0):
    """Greedy Markov walk recomputed with numpy/torch routines (matmul, argmax, bf16 conversion)."""
    Wf = bf16_vals(W).astype(np.float64)
    Ef = bf16_vals(E)
    B, G, V = base.shape
    toks = np.zeros((B, G), np.int64)
    zs = np.zeros((B, G, V), np.float32)
    for b in range(B):
        s = s0[b].astype(np.float32)
        for t in range(G):
            q = lib_bf16_round_f32(s).astype(np.float64)
            z = (Wf @ q).astype(np.float32) + base[b, t]
            zs[b, t] = z
            toks[b, t] = int(np.argmax(z))        # numpy returns the first maximum
            s = Ef[toks[b, t]]
    return toks, zs


@pytest.mark.parametrize("seed", range(100))
def test_bruteforce_fig2_shape(seed):
    d = I.make_inputs(MARKOV, V=12, r=4, B=2, gamma=3, seed=seed)
    out = O.walk(MARKOV, d["W"], d["E"], d["base"], d["s0"], want_z=True)
    toks, zs = rederive_markov(d["W"], d["E"], d["base"], d["s0"])
    np.testing.assert_array_equal(out["tokens"], toks)
    # fp64 sums in a different order can differ in the last fp64 bits; after rounding to fp32 they agree
    np.testing.assert_allclose(out["z"], zs, rtol=0, atol=1e-6)


@pytest.mark.parametrize("V,r,B,G", [(64, 16, 3, 5), (257, 32, 2, 4), (1000, 64, 1, 6)])
def test_projection_matches_library_matmul(V, r, B, G):
    d = I.make_inputs(MARKOV, V, r, B, G, seed=7)
    out = O.walk(MARKOV, d["W"], d["E"], d["base"], d["s0"], want_z=True, want_logits=True)
    toks, zs = rederive_markov(d["W"], d["E"], d["base"], d["s0"])
    np.testing.assert_array_equal(out["tokens"], toks)
    np.testing.assert_allclose(out["z"], zs, rtol=0, atol=1e-6)
    # the emitted logits are the single bf16 rounding of z (torch conversion as the library reference)
    np.testing.assert_array_equal(bf16_vals(out["logits"]), lib_bf16_round_f32(out["z"]))


def test_gap_is_top1_minus_top2():
    d = I.make_inputs(MARKOV, 500, 32, 2, 4, seed=3)
    out = O.walk(MARKOV, d["W"], d["E"], d["base"], d["s0"], want_z=True)
    srt = np.sort(out["z"], axis=-1)
    np.testing.assert_allclose(out["gap"], (srt[..., -1].astype(np.float64) - srt[..., -2]), rtol=0, atol=1e-6)


# ---------------------------------------------------------------------------------------------
# 3. Special cases that reduce to textbook routines.
# ---------------------------------------------------------------------------------------------
def test_zero_projection_is_argmax_of_base():
    d = I.make_inputs(MARKOV, 300, 16, 3, 5, seed=11)
    W0 = np.zeros_like(d["W"])
    out = O.walk(MARKOV, W0, d["E"], d["base"], d["s0"])
    np.testing.assert_array_equal(out["tokens"], np.argmax(d["base"], axis=-1))


def test_zero_embedding_markov_later_steps_argmax_base():
    d = I.make_inputs(MARKOV, 300, 16, 2, 5, seed=12)
    E0 = np.zeros_like(d["E"])
    out = O.walk(MARKOV, d["W"], E0, d["base"], d["s0"])
    np.testing.assert_array_equal(out["tokens"][:, 1:], np.argmax(d["base"][:, 1:], axis=-1))


def test_batch_rows_are_independent_walks():
    d = I.make_inputs(MARKOV, 400, 32, 4, 6, seed=13)
    full = O.walk(MARKOV, d["W"], d["E"], d["base"], d["s0"], T=1.0, seed=99)
    for b in range(4):
        # walk b alone must carry its batch index into the noise counter: emulate with a padded batch
        pad_base = np.zeros((b + 1, 6, 400), np.float32)
        pad_base[b] = d["base"][b]
        pad_s0 = np.zeros((b + 1, 32), np.float32)
        pad_s0[b] = d["s0"][b]
        one = O.walk(MARKOV, d["W"], d["E"], pad_base, pad_s0, T=1.0, seed=99)
        np.testing.assert_array_equal(one["tokens"][b], full["tokens"][b])
    greedy = O.walk(MARKOV, d["W"], d["E"], d["base"], d["s0"])
    for b in range(4):
        one = O.walk(MARKOV, d["W"], d["E"], d["base"][b:b + 1], d["s0"][b:b + 1])
        np.testing.assert_array_equal(one["tokens"][0], greedy["tokens"][b])


def test_recurrent_state_matches_library_tanh():
    d = I.make_inputs(RECURRENT, 300, 32, 2, 5, seed=14)
    c = I.normal_f32(5, "A", (32,), 0.1)
    out = O.walk(RECURRENT, d["W"], d["E"], d["base"], d["s0"], A=d["A"], c=c, want_state=True, want_z=True)
    Wf = bf16_vals(d["W"]).astype(np.float64)
    Ef = bf16_vals(d["E"]).astype(np.float64)
    A = d["A"].astype(np.float64)
    for b in range(2):
        h = d["s0"][b].astype(np.float32)
        for t in range(5):
            z = (Wf @ lib_bf16_round_f32(h).astype(np.float64)).astype(np.float32) + d["base"][b, t]
            x = int(np.argmax(z))
            assert out["tokens"][b, t] == x
            h = np.tanh(A @ h.astype(np.float64) + Ef[x] + c.astype(np.float64)).astype(np.float32)
            np.testing.assert_allclose(out["state"][b, t], h, rtol=0, atol=2e-7)


# ---------------------------------------------------------------------------------------------
# 4. Ties: the smallest index wins; -0 equals +0.
# ---------------------------------------------------------------------------------------------
def test_ties_lowest_index_and_signed_zero():
    V, r = 8, 16
    W0 = np.zeros((V, r), np.uint16)
    E = np.zeros((V, r), np.uint16)
    base = np.full((1, 3, V), -1.0, np.float32)
    base[0, 0, [2, 5, 6]] = 0.75                   # equal maxima -> 2
    base[0, 1, 1] = -0.0                           # -0 and +0 tie -> 1
    base[0, 1, 3] = 0.0
    base[0, 2, 7] = 0.5                            # unique maximum at the last row
    out = O.walk(MARKOV, W0, E, base, np.zeros((1, r), np.float32))
    assert out["tokens"].tolist() == [[2, 1, 7]]
    assert out["gap"][0, 0] == 0.0 and out["gap"][0, 1] == 0.0


# ---------------------------------------------------------------------------------------------
# 5. Resume invariance: re-running from any step with the state reached there reproduces the rest.
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("kind,T", [(MARKOV, 0.0), (MARKOV, 1.0), (RECURRENT, 0.0), (RECURRENT, 0.7)])
def test_resume_from_any_step(kind, T):
    G = 7
    d = I.make_inputs(kind, 600, 32, 2, G, seed=21)
    full = O.walk(kind, d["W"], d["E"], d["base"], d["s0"], A=d["A"], c=d["c"], T=T, seed=5, want_state=True,
                  want_z=True)
    for t0 in range(1, G):
        part = O.walk(kind, d["W"], d["E"], np.ascontiguousarray(d["base"][:, t0:]),
                      np.ascontiguousarray(full["state"][:, t0 - 1]), A=d["A"], c=d["c"], t0=t0, T=T, seed=5,
                      want_state=True, want_z=True)
        np.testing.assert_array_equal(part["tokens"], full["tokens"][:, t0:])
        np.testing.assert_array_equal(part["state"], full["state"][:, t0:])
        np.testing.assert_array_equal(part["z"], full["z"][:, t0:])


# ---------------------------------------------------------------------------------------------
# 6. Rounding and the noise generator.
# ---------------------------------------------------------------------------------------------
def test_bf16_round_matches_torch_including_ties():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(10.0)
    # exact halfway cases: low 16 bits = 0x8000, with both parities of the kept bit
    hw = (rng.integers(0x3F00, 0x4100, 2000).astype(np.uint32) << 16) | 0x8000
    x = np.concatenate([x, hw.view(np.float32), -hw.view(np.float32), np.float32([0.0, -0.0, 1e-40, 3e38])])
    ours = np.array([O.bf16_round(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(ours, bf16_bits(x))


def test_philox_known_answers():
    # Philox4x32-10 known-answer vectors published with the SC'11 Random123 release
    assert O.philox4x32_10([0, 0, 0, 0], [0, 0]) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert O.philox4x32_10([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2) == [0x408F276D, 0x41C83B0E, 0xA20BC7C6,
                                                                    0x6D5451FD]
    assert O.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0]) == \
        [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_philox_matches_triton_library():
    """Compare with triton's Philox (tl.philox, 10 rounds) run by triton's CPU interpreter."""
    import os
    import subprocess
    import sys
    pytest.importorskip("triton")
    rng = np.random.default_rng(1)
    ctr = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64)
    key = rng.integers(0, 2**32, size=(2,), dtype=np.uint64)
    script = r'''
import sys, json, numpy as np, torch, triton, triton.language as tl
@triton.jit
def k(c0p, c1p, c2p, c3p, out, seed, N: tl.constexpr):
    i = tl.arange(0, N)
    a, b, c, d = tl.philox(seed, tl.load(c0p + i), tl.load(c1p + i), tl.load(c2p + i), tl.load(c3p + i), 10)
    tl.store(out + 4 * i, a); tl.store(out + 4 * i + 1, b); tl.store(out + 4 * i + 2, c); tl.store(out + 4 * i + 3, d)
inp = json.loads(sys.stdin.read())
ctr = np.array(inp["ctr"], dtype=np.int64)
cols = [torch.tensor(ctr[:, j]).to(torch.uint32).contiguous() for j in range(4)]
out = torch.zeros(4 * ctr.shape[0], dtype=torch.uint32)
k[(1,)](cols[0], cols[1], cols[2], cols[3], out, inp["seed"], N=ctr.shape[0])
print(json.dumps([int(x) for x in out.to(torch.int64)]))
'''
    import json
    seed = int(key[0]) | (int(key[1]) << 32)
    env = dict(os.environ, TRITON_INTERPRET="1")
    res = subprocess.run([sys.executable, "-c", script], input=json.dumps({"ctr": ctr.tolist(), "seed": seed}),
                         capture_output=True, text=True, env=env, timeout=600)
    if res.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + res.stderr.strip().splitlines()[-1][:200])
    theirs = json.loads(res.stdout.strip().splitlines()[-1])
    ours = []
    for row in ctr:
        ours += O.philox4x32_10([int(v) for v in row], [int(key[0]), int(key[1])])
    assert ours == theirs


def test_uniform_is_exact_and_open():
    for w in [0, 1, 511, 512, 0x80000000, 0xFFFFFE00, 0xFFFFFFFF, 0x12345678]:
        u = O.uniform(w)
        exact = (Fraction(w >> 9) + Fraction(1, 2)) / 2**23
        assert Fraction(u) == exact
        assert 0.0 < u < 1.0
    assert O.uniform(0) == 2.0**-24 and O.uniform(0xFFFFFFFF) == 1.0 - 2.0**-24


def test_noise_words_uniform_chi2():
    words = np.array([O.noise_word(123, b, tau, v) for b in range(2) for tau in range(4) for v in range(2048)],
                     dtype=np.uint64)
    counts = np.bincount((words >> 28).astype(np.int64), minlength=16)
    n = words.size
    chi2 = float(((counts - n / 16) ** 2 / (n / 16)).sum())
    assert chi2 < 45.0        # 15 degrees of freedom: p < 1e-4 above 45
    # counter layout: rows 4k..4k+3 share a counter and take its four words in order
    w4 = O.philox4x32_10([5, 3, 1, 0], [123, 0])
    assert [O.noise_word(123, 1, 3, 20 + j) for j in range(4)] == w4


def test_gumbel_moments_closed_form():
    g = np.array([O.gumbel(7, 0, 0, v) for v in range(200000)], np.float64)
    euler_gamma = 0.5772156649015329
    assert abs(g.mean() - euler_gamma) < 5 * math.sqrt(math.pi**2 / 6 / g.size)
    assert abs(g.var() - math.pi**2 / 6) < 0.03


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_gumbel_max_sampling_law(T):
    """Sampled tokens follow softmax(z / T) (Gumbel-max), within 5 binomial sigmas."""
    V, r, n = 8, 16, 40000
    z = np.array([0.0, 1.0, -0.5, 2.0, 0.3, -1.0, 1.5, 0.0], np.float32)
    base = np.broadcast_to(z, (n, 1, V)).copy()
    out = O.walk(MARKOV, np.zeros((V, r), np.uint16), np.zeros((V, r), np.uint16), base,
                 np.zeros((n, r), np.float32), T=T, seed=2024)
    freq = np.bincount(out["tokens"][:, 0], minlength=V) / n
    p = np.exp(z.astype(np.float64) / T)
    p /= p.sum()
    sigma = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(freq - p) < 5 * sigma + 1e-12), (freq, p)


def test_invalid_arguments_rejected():
    W, E, base, s0 = hand_inputs()
    with pytest.raises(ValueError):
        O.walk(RECURRENT, W, E, base, s0)          # recurrent head without A
    with pytest.raises(ValueError):
        O.walk(MARKOV, W, E, base, s0, T=-1.0)


def test_walk_prefix_is_the_shorter_walk():
    """A walk's first steps do not depend on later base logits (Fig. 2: each step uses only the state the
    earlier steps produced): the first g steps of a gamma-step walk equal the g-step walk, sampled or not."""
    for kind, T in ((MARKOV, 0.0), (MARKOV, 1.0), (RECURRENT, 0.7)):
        d = I.make_inputs(kind, 300, 32, 3, 7, seed=21)
        full = O.walk(kind, d["W"], d["E"], d["base"], d["s0"], A=d["A"], c=d["c"], T=T, seed=4, want_state=True)
        for g in (1, 3):
            part = O.walk(kind, d["W"], d["E"], np.ascontiguousarray(d["base"][:, :g]), d["s0"], A=d["A"], c=d["c"],
                          T=T, seed=4, want_state=True)
            np.testing.assert_array_equal(part["tokens"], full["tokens"][:, :g])
            np.testing.assert_array_equal(part["state"], full["state"][:, :g])


@pytest.mark.parametrize("kind,T,e4m3", [(MARKOV, 0.0, False), (MARKOV, 1.0, False), (RECURRENT, 0.7, False),
                                          (MARKOV, 1.0, True)])
def test_thread_count_does_not_change_results(kind, T, e4m3):
    """The oracle may split a step's rows over threads (OpenMP); every output must be bit-identical to the
    single-threaded walk."""
    d = I.make_inputs(kind, 5003, 128, 2, 4, seed=8)
    w8 = O.quantize_w_e4m3(d["W"]) if e4m3 else None
    kw = dict(A=d["A"], c=d["c"], T=T, seed=3, want_logits=True, want_z=True, want_gap=True, want_state=True,
              w_e4m3=w8)
    try:
        assert O.set_threads(1) == 1
        one = O.walk(kind, d["W"], d["E"], d["base"], d["s0"], **kw)
        n = O.set_threads(4)
        many = O.walk(kind, d["W"], d["E"], d["base"], d["s0"], **kw)
    finally:
        O.set_threads(1)
    print(f"threads used: {n}")
    for k in one:
        np.testing.assert_array_equal(one[k], many[k], err_msg=k)
