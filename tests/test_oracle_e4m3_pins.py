"""Pins of the oracle's E4M3 path (weights as E4M3 codes with a per-row scale, the state as two scaled E4M3
vectors; the pages' Fig. 7 design restated with the 8-bit float format). Every check compares the oracle with
something other than itself: the library's own E4M3 conversion, error bounds that follow from the format,
brute force with a library matmul, and the special case in which the E4M3 walk must equal the bf16 walk."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
import whead_inputs as I

MARKOV, RECURRENT = O.MARKOV, O.RECURRENT
NAN_CODES = (0x7F, 0xFF)


def torch_codes(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e4m3_grid():
    """Every finite non-negative E4M3 value, ascending (from the library's decoding)."""
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def test_decoding_matches_library():
    for code in range(256):
        if code in NAN_CODES:
            assert np.isnan(O.e4m3_value(code))
            continue
        want = float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).float()[0])
        assert O.e4m3_value(code) == want, hex(code)
    assert O.e4m3_value(0x7E) == 448.0 and O.e4m3_value(0x01) == 2.0 ** -9 and O.e4m3_value(0x08) == 2.0 ** -6


def test_rounding_matches_library_including_ties_and_subnormals():
    rng = np.random.default_rng(7)
    grid = e4m3_grid()
    mids = (grid[1:] + grid[:-1]) / 2  # exact ties: each must go to the even mantissa
    rand = np.exp2(rng.uniform(-12, np.log2(440), 20000)) * rng.choice([-1, 1], 20000)
    xs = np.concatenate([grid, -grid, mids, -mids, rand, [0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -11, 447.9]])
    xs = xs.astype(np.float32)
    got = np.array([O.e4m3_round(float(x)) for x in xs], dtype=np.uint8)
    np.testing.assert_array_equal(got, torch_codes(xs))


def test_rounding_saturates_above_the_largest_value():
    assert O.e4m3_round(448.0) == 0x7E and O.e4m3_round(460.0) == 0x7E and O.e4m3_round(1e6) == 0x7E
    assert O.e4m3_round(-1e6) == 0xFE


@pytest.mark.parametrize("n", [1, 7, 256])
def test_vector_quantization_bounds(n):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * np.exp2(rng.uniform(-8, 8))).astype(np.float32)
    s, q = O.quantize_e4m3(x)
    assert s == np.float32(np.float32(np.abs(x).max()) / np.float32(448.0))
    vals = np.array([O.e4m3_value(c) for c in q])
    # the largest magnitude maps to +-448, and every element is within half a spacing of the format
    assert np.abs(vals[np.argmax(np.abs(x))]) == 448.0
    grid = e4m3_grid()
    xs = x.astype(np.float64) / s
    spacing = np.array([grid[min(np.searchsorted(grid, abs(t)), len(grid) - 1)] - grid[max(np.searchsorted(grid, abs(t)) - 1, 0)]
                        for t in xs])
    assert np.all(np.abs(xs - vals) <= spacing / 2 + 1e-6 * np.abs(xs))


def test_zero_vector_quantizes_to_zero_scale():
    s, q = O.quantize_e4m3(np.zeros(16, dtype=np.float32))
    assert s == 0.0 and not q.any()


def test_two_vector_split_error_bound():
    """hi captures u to within s1 * 16 (half the largest spacing, 32); lo captures that residual to within
    s2 * 16; so |u - s1 hi - s2 lo| <= max|u| / 784."""
    rng = np.random.default_rng(3)
    for _ in range(50):
        u = (rng.standard_normal(256) * np.exp2(rng.uniform(-6, 6))).astype(np.float32)
        s1, hi, s2, lo = O.split_e4m3(u)
        rec = s1 * np.array([O.e4m3_value(c) for c in hi]) + s2 * np.array([O.e4m3_value(c) for c in lo])
        assert np.max(np.abs(u - rec)) <= np.abs(u).max() / 784 * (1 + 1e-5)


def test_two_vector_split_of_a_representable_state_is_exact():
    grid = e4m3_grid()
    rng = np.random.default_rng(4)
    vals = rng.choice(np.concatenate([grid, -grid]), 64)
    vals[5] = 448.0
    u = (vals * 2.0 ** -5).astype(np.float32)  # power-of-two scale: exact in fp32
    s1, hi, s2, lo = O.split_e4m3(u)
    assert s1 == 2.0 ** -5 and s2 == 0.0 and not lo.any()
    np.testing.assert_array_equal(np.array([O.e4m3_value(c) for c in hi], dtype=np.float32) * np.float32(s1), u)


def test_weight_quantization_is_rowwise_vector_quantization():
    d = I.make_inputs(MARKOV, 37, 32, 1, 1, seed=2)
    Wq, sw = O.quantize_w_e4m3(d["W"])
    Wf = I.bf16_to_f32(d["W"]) if hasattr(I, "bf16_to_f32") else (d["W"].astype(np.uint32) << 16).view(np.float32)
    for v in range(37):
        s, q = O.quantize_e4m3(Wf[v])
        assert sw[v] == s
        np.testing.assert_array_equal(Wq[v], q)


def brute_force_e4m3(kind, Wq, sw, E, base, s0, A=None):
    """The E4M3 walk re-derived with a library matmul (greedy): dequantized codes in fp64."""
    dec = np.array([O.e4m3_value(c) if c not in NAN_CODES else 0.0 for c in range(256)])
    Wd = dec[Wq]
    Ef = (E.astype(np.uint32) << 16).view(np.float32)
    B, G, V = base.shape
    toks = np.zeros((B, G), dtype=np.int32)
    for b in range(B):
        s = s0[b].astype(np.float32)
        for t in range(G):
            s1, hi, s2, lo = O.split_e4m3(s)
            p = sw.astype(np.float64) * (s1 * (Wd @ dec[hi]) + s2 * (Wd @ dec[lo]))
            z = p.astype(np.float32) + base[b, t]
            x = int(np.argmax(z))
            toks[b, t] = x
            s = Ef[x].copy() if kind == MARKOV else np.tanh(A.astype(np.float64) @ s + Ef[x]).astype(np.float32)
    return toks


@pytest.mark.parametrize("seed", range(20))
def test_e4m3_walk_matches_brute_force(seed):
    d = I.make_inputs(MARKOV, 48, 16, 2, 4, seed=100 + seed)
    Wq, sw = O.quantize_w_e4m3(d["W"])
    ref = O.walk(MARKOV, d["W"], d["E"], d["base"], d["s0"], w_e4m3=(Wq, sw))
    np.testing.assert_array_equal(ref["tokens"], brute_force_e4m3(MARKOV, Wq, sw, d["E"], d["base"], d["s0"]))


def test_e4m3_walk_equals_bf16_walk_when_everything_is_representable():
    """W rows and E rows that are power-of-two multiples of E4M3 values (each row reaching 448 times its
    scale) quantize exactly, and the state splits exactly; the projection is then the same exact sum, so the
    E4M3 walk and the bf16 walk give the same z and tokens."""
    rng = np.random.default_rng(9)
    grid = e4m3_grid()
    V, r, B, G = 200, 32, 2, 5
    def rows(scale_exp):
        vals = rng.choice(np.concatenate([grid[8:], -grid[8:]]), (V, r))
        vals[:, 0] = 448.0 * rng.choice([-1, 1], V)
        f = (vals * np.exp2(scale_exp)).astype(np.float32)
        return (f.view(np.uint32) >> 16).astype(np.uint16), f
    W, Wf = rows(-12)
    E, Ef = rows(-8)
    assert np.array_equal(((W.astype(np.uint32) << 16).view(np.float32)), Wf)  # bf16-exact
    base = (rng.standard_normal((B, G, V)) * 2).astype(np.float32)
    s0 = Ef[rng.integers(0, V, B)].copy()
    Wq, sw = O.quantize_w_e4m3(W)
    assert np.all(sw == np.float32(2.0 ** -12))
    a = O.walk(MARKOV, W, E, base, s0, want_z=True)
    b = O.walk(MARKOV, W, E, base, s0, want_z=True, w_e4m3=(Wq, sw))
    np.testing.assert_array_equal(a["z"], b["z"])
    np.testing.assert_array_equal(a["tokens"], b["tokens"])


@pytest.mark.parametrize("kind,T", [(MARKOV, 0.0), (MARKOV, 1.0), (RECURRENT, 0.0)])
def test_e4m3_walk_resume_from_any_step(kind, T):
    d = I.make_inputs(kind, 300, 32, 2, 6, seed=5)
    Wq, sw = O.quantize_w_e4m3(d["W"])
    full = O.walk(kind, d["W"], d["E"], d["base"], d["s0"], A=d["A"], c=d["c"], T=T, seed=11, want_z=True,
                  want_state=True, w_e4m3=(Wq, sw))
    for t0 in range(1, 6):
        part = O.walk(kind, d["W"], d["E"], d["base"][:, t0:].copy(), full["state"][:, t0 - 1].copy(), A=d["A"],
                      c=d["c"], T=T, seed=11, t0=t0, want_z=True, want_state=True, w_e4m3=(Wq, sw))
        np.testing.assert_array_equal(part["tokens"], full["tokens"][:, t0:])
        np.testing.assert_array_equal(part["z"], full["z"][:, t0:])


def test_vectors_below_the_normal_range_quantize_to_zero():
    """448 * FLT_MIN is the smallest largest-magnitude with a finite reciprocal scale; below it the vector is
    taken as zero (scale 0, zero codes), at it the scale is exactly FLT_MIN."""
    tiny = np.float32(448.0) * np.float32(np.finfo(np.float32).tiny)
    s, q = O.quantize_e4m3(np.array([tiny * np.float32(0.5), -tiny * np.float32(0.25)], dtype=np.float32))
    assert s == 0.0 and not q.any()
    s, q = O.quantize_e4m3(np.array([tiny, 0.0], dtype=np.float32))
    assert s == np.finfo(np.float32).tiny and q[0] == 0x7E
