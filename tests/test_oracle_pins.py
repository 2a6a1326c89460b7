"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against something fixed independently of it:
the hand-worked example (tests/golden), brute-force loops on tiny inputs,
library conversions (numpy's float16, torch's GELU), closed forms and
mathematical identities, and exact integer arithmetic.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

EPIS = ["none", "bias", "relu_bias", "gelu_bias", "relu_aux_bias"]


def f16_bits(x):
    return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)


def plain_to_layout(Aplain, Bplain, a_major, b_major):
    """Lay the plain matrices A[M][K], B[K][N] out as the oracle reads them."""
    A = Aplain if a_major == "k" else Aplain.T
    B = Bplain.T if b_major == "k" else Bplain
    return np.ascontiguousarray(A).reshape(-1), np.ascontiguousarray(B).reshape(-1)


# ---------------------------------------------------------------- fp16 codec

def test_f16_decode_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.f16_decode(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, got[0x8000]) == -1.0


def test_f16_encode_roundtrip_all_finite(oracle):
    bits = np.arange(65536, dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(vals)
    assert np.array_equal(oracle.f16_encode(vals[fin]), bits[fin])


def test_f16_encode_ties_and_neighbours(oracle):
    # Midpoints between consecutive positive finite halves round to the even
    # neighbour; one double-ulp either side rounds to the nearer one.
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)
    a = lo.view(np.float16).astype(np.float64)
    b = (lo + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mid = (a + b) / 2  # exact in fp64
    even = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(oracle.f16_encode(mid), even)
    assert np.array_equal(oracle.f16_encode(np.nextafter(mid, 0)), lo)
    assert np.array_equal(oracle.f16_encode(np.nextafter(mid, np.inf)), (lo + 1).astype(np.uint16))
    # negative side mirrors the positive side
    assert np.array_equal(oracle.f16_encode(-mid), even | 0x8000)


def test_f16_encode_boundaries(oracle):
    enc = lambda x: int(oracle.f16_encode(np.array([x]))[0])
    assert enc(65504.0) == 0x7BFF
    assert enc(65519.999) == 0x7BFF
    assert enc(65520.0) == 0x7C00          # tie to even -> overflow
    assert enc(-70000.0) == 0xFC00
    assert enc(math.inf) == 0x7C00
    assert enc(2.0 ** -24) == 0x0001       # smallest subnormal
    assert enc(2.0 ** -25) == 0x0000       # tie to even -> zero
    assert enc(3 * 2.0 ** -25) == 0x0002   # 1.5 ulp -> 2 (even)
    assert enc(2.0 ** -14) == 0x0400       # smallest normal
    assert enc(2.0 ** -14 - 2.0 ** -26) == 0x0400  # rounds up into the normals
    assert enc(-0.0) == 0x8000
    assert enc(math.nan) & 0x7C00 == 0x7C00 and enc(math.nan) & 0x3FF


def test_f16_encode_random_vs_numpy(oracle):
    rng = np.random.default_rng(7)
    mag = np.exp2(rng.uniform(-30, 15.99, 200000))
    x = mag * rng.choice([-1.0, 1.0], mag.size)
    ref = x.astype(np.float16).view(np.uint16)  # numpy rounds fp64 -> fp16 to nearest even
    assert np.array_equal(oracle.f16_encode(x), ref)


# ------------------------------------------------------------- hand-worked

def test_hand_worked_example(oracle):
    g = json.load(open(os.path.join(GOLDEN, "hand_2x3x4.json")))
    M, N, K = g["M"], g["N"], g["K"]
    A = f16_bits(g["A"]).reshape(-1)
    B = f16_bits(g["B"]).reshape(-1)
    bias = f16_bits(g["bias"])
    # NONE: the plain product
    r = oracle.linear_forward(A, B, None, "none", M, N, K, a_major="k", b_major="n", d_layout="row")
    assert np.array_equal(r["Z"].reshape(M, N), np.array(g["AB"], float))
    # BIAS: product plus bias broadcast over columns
    r = oracle.linear_forward(A, B, bias, "bias", M, N, K, a_major="k", b_major="n")
    assert np.array_equal(r["Z"].reshape(M, N), np.array(g["Z"], float))
    assert np.array_equal(oracle.f16_decode(r["D"]).reshape(M, N), np.array(g["Z"], float))
    # RELU_AUX_BIAS: ReLU values and the bit-packed mask
    r = oracle.linear_forward(A, B, bias, "relu_aux_bias", M, N, K, a_major="k", b_major="n")
    assert np.array_equal(oracle.f16_decode(r["D"]).reshape(M, N), np.array(g["relu"], float))
    assert r["ld_aux"] == 4
    assert r["aux"].tolist() == g["mask_words_row_major_ld4"]
    # DRELU_BGRAD
    dY = f16_bits(g["dY"]).reshape(-1)
    dZ, bgrad = oracle.drelu_bgrad(dY, r["aux"], M, N, d_layout="row")
    assert np.array_equal(oracle.f16_decode(dZ).reshape(M, N), np.array(g["dZ"], float))
    assert bgrad.tolist() == g["bgrad"]


def test_hand_worked_example_all_layouts(oracle):
    """The same example read through every operand/output layout."""
    g = json.load(open(os.path.join(GOLDEN, "hand_2x3x4.json")))
    M, N, K = g["M"], g["N"], g["K"]
    Ap = np.array(g["A"], float)
    Bp = np.array(g["B"], float)
    for am in "km":
        for bm in "kn":
            for dl in ("row", "col"):
                A, B = plain_to_layout(f16_bits(Ap).reshape(M, K), f16_bits(Bp).reshape(K, N), am, bm)
                r = oracle.linear_forward(A, B, f16_bits(g["bias"]), "relu_aux_bias", M, N, K,
                                          a_major=am, b_major=bm, d_layout=dl)
                Z = r["Z"].reshape((M, N) if dl == "row" else (N, M))
                if dl == "col":
                    Z = Z.T
                assert np.array_equal(Z, np.array(g["Z"], float)), (am, bm, dl)
                rows, cols = (M, N) if dl == "row" else (N, M)
                words = r["aux"].reshape(rows, r["ld_aux"])
                bits = np.array([[(words[i, j // 32] >> (j % 32)) & 1 for j in range(cols)]
                                 for i in range(rows)])
                if dl == "col":
                    bits = bits.T
                assert bits.tolist() == g["mask_rows"], (am, bm, dl)


# ------------------------------------------------------------ brute force

def _brute(Aplain, Bplain, bias, epi):
    """Pure-Python triple loop on the plain matrices (tiny sizes only)."""
    M, K = Aplain.shape
    N = Bplain.shape[1]
    Z = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += float(Aplain[m, k]) * float(Bplain[k, n])
            if epi != "none":
                s += float(bias[m])
            Z[m, n] = s
    zt = torch.from_numpy(Z)
    if epi in ("relu_bias", "relu_aux_bias"):
        Y = torch.relu(zt).numpy()
    elif epi == "gelu_bias":
        Y = torch.nn.functional.gelu(zt, approximate="tanh").numpy()
    else:
        Y = Z
    return Z, Y


@pytest.mark.parametrize("am,bm,dl", [(a, b, d) for a in "km" for b in "kn" for d in ("row", "col")])
def test_brute_force_tiny(oracle, am, bm, dl):
    rng = np.random.default_rng(100 + "km".index(am) * 4 + "kn".index(bm) * 2 + (dl == "col"))
    for M in range(1, 6):
        for N in range(1, 6):
            for K in (1, 2, 3, 5, 8):
                epi = EPIS[(M + N + K) % len(EPIS)]
                Ap = rng.standard_normal((M, K)).astype(np.float16)
                Bp = rng.standard_normal((K, N)).astype(np.float16)
                bias = rng.standard_normal(M).astype(np.float16)
                A, B = plain_to_layout(Ap.view(np.uint16), Bp.view(np.uint16), am, bm)
                r = oracle.linear_forward(A, B, bias.view(np.uint16), epi, M, N, K,
                                          a_major=am, b_major=bm, d_layout=dl, threads=1)
                Z, Y = _brute(Ap.astype(np.float64), Bp.astype(np.float64),
                              bias.astype(np.float64), epi)
                shape = (M, N) if dl == "row" else (N, M)
                Zo = r["Z"].reshape(shape)
                Do = r["D"].reshape(shape)
                if dl == "col":
                    Zo, Do = Zo.T, Do.T
                assert np.array_equal(Zo, Z), (M, N, K, epi)
                assert np.array_equal(Do, Y.astype(np.float16).view(np.uint16)), (M, N, K, epi)


def test_padded_leading_dimensions(oracle):
    """Leading dimensions larger than the logical extent are honoured."""
    rng = np.random.default_rng(3)
    M, N, K = 5, 7, 9
    Ap = rng.standard_normal((M, K)).astype(np.float16)
    Bp = rng.standard_normal((K, N)).astype(np.float16)
    lda, ldb, ldd = K + 3, K + 5, M + 8
    A = np.full((M, lda), np.float16(np.nan))
    A[:, :K] = Ap
    B = np.full((N, ldb), np.float16(np.nan))  # K-major B: row n holds B[:, n]
    B[:, :K] = Bp.T
    r = oracle.linear_forward(A.view(np.uint16).reshape(-1), B.view(np.uint16).reshape(-1), None,
                              "none", M, N, K, a_major="k", b_major="k", d_layout="col",
                              lda=lda, ldb=ldb, ldd=ldd)
    Z = r["Z"].reshape(N, ldd)[:, :M].T
    assert np.array_equal(Z, _brute(Ap.astype(float), Bp.astype(float), None, "none")[0])


# ------------------------------------------------------------------ GELU

def test_gelu_closed_forms(oracle):
    act = lambda z: oracle.act_f64("gelu_bias", z)
    assert act(0.0) == 0.0
    # published value of the tanh approximation at 1
    assert abs(act(1.0) - 0.8411919906082768) < 1e-15
    # large |z|: identity above, zero below
    assert act(12.0) == 12.0
    assert abs(act(-12.0)) < 1e-40
    for z in np.linspace(-6, 6, 241):
        # GELU(z) - GELU(-z) = z holds for the tanh form exactly in real arithmetic
        assert abs(act(z) - act(-z) - z) <= 4e-16 * max(1.0, abs(z))


def test_gelu_sigmoid_identity(oracle):
    """0.5(1 + tanh(u)) = 1/(1 + exp(-2u)): an independent way to evaluate it."""
    c = math.sqrt(2.0 / math.pi)
    for z in np.linspace(-8, 8, 1601):
        u = c * (z + 0.044715 * z ** 3)
        ref = z / (1.0 + math.exp(-2.0 * u))
        assert abs(oracle.act_f64("gelu_bias", z) - ref) <= 1e-14 * max(1.0, abs(z))


def test_gelu_close_to_exact_erf_gelu(oracle):
    """The tanh form approximates z*Phi(z) to within about 5e-4 everywhere."""
    worst = 0.0
    for z in np.linspace(-10, 10, 4001):
        exact = 0.5 * z * (1.0 + math.erf(z / math.sqrt(2.0)))
        worst = max(worst, abs(oracle.act_f64("gelu_bias", z) - exact))
    assert worst < 1e-3
    assert worst > 1e-5  # it is the approximation, not the erf form


def test_gelu_matches_torch_tanh_gelu(oracle):
    z = torch.linspace(-9, 9, 7001, dtype=torch.float64)
    ref = torch.nn.functional.gelu(z, approximate="tanh").numpy()
    got = np.array([oracle.act_f64("gelu_bias", float(v)) for v in z])
    # 1 + tanh(u) cancels for very negative z in both evaluations, so values
    # below ~1e-15 in magnitude are rounding noise (far below fp16's 6e-8).
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-15)


def test_relu_and_none(oracle):
    for z in (-3.5, -0.0, 0.0, 1e-30, 2.25):
        assert oracle.act_f64("relu_bias", z) == max(z, 0.0)
        assert oracle.act_f64("relu_aux_bias", z) == max(z, 0.0)
        assert oracle.act_f64("bias", z) == z
        assert oracle.act_f64("none", z) == z


# ------------------------------------------------------ mask / relu identity

def test_relu_equals_z_times_mask(oracle):
    rng = np.random.default_rng(11)
    M, N, K = 37, 70, 24
    A = rng.standard_normal(M * K).astype(np.float16)
    B = rng.standard_normal(K * N).astype(np.float16)
    bias = rng.standard_normal(M).astype(np.float16)
    for dl in ("row", "col"):
        rb = oracle.linear_forward(A, B, bias, "bias", M, N, K, d_layout=dl)
        rr = oracle.linear_forward(A, B, bias, "relu_aux_bias", M, N, K, d_layout=dl)
        rows, cols = (M, N) if dl == "row" else (N, M)
        ld_aux = rr["ld_aux"]
        assert ld_aux == 4 * ((cols + 127) // 128)
        words = rr["aux"].reshape(rows, ld_aux)
        bits = np.zeros((rows, ld_aux * 32), np.int64)
        for j in range(ld_aux * 32):
            bits[:, j] = (words[:, j // 32] >> np.uint32(j % 32)) & 1
        assert not bits[:, cols:].any()  # padding bits are zero
        bits = bits[:, :cols].reshape(-1)
        z = rb["Z"]
        assert np.array_equal(bits, (z > 0).astype(np.int64))
        y_bias = oracle.f16_decode(rb["D"])
        y_relu = oracle.f16_decode(rr["D"])
        assert np.array_equal(y_relu, y_bias * bits)


# ------------------------------------------------------- exact integer case

@pytest.mark.parametrize("M,N,K", [(64, 48, 128), (19, 17, 128)])
def test_exact_integer_case(oracle, M, N, K):
    """Integer entries keep every partial sum exact in fp16 inputs, fp32 and
    fp16 outputs; the oracle must equal integer matrix arithmetic."""
    rng = np.random.default_rng(M * 1000 + N)
    Ai = rng.integers(-2, 3, (M, K))
    Bi = rng.integers(-2, 3, (K, N))
    bi = rng.integers(-8, 9, M)
    exact = Ai @ Bi + bi[:, None]
    assert np.abs(exact).max() < 2048
    for epi in ("bias", "relu_bias", "relu_aux_bias"):
        r = oracle.linear_forward(f16_bits(Ai).reshape(-1), f16_bits(Bi).reshape(-1), f16_bits(bi),
                                  epi, M, N, K, a_major="k", b_major="n")
        assert np.array_equal(r["Z"].reshape(M, N), exact.astype(float))
        y = exact if epi == "bias" else np.maximum(exact, 0)
        assert np.array_equal(r["D"].reshape(M, N), f16_bits(y))


def test_none_matches_library_matmul(oracle):
    rng = np.random.default_rng(5)
    M, N, K = 33, 29, 64
    Ap = rng.standard_normal((M, K)).astype(np.float16)
    Bp = rng.standard_normal((K, N)).astype(np.float16)
    A, B = plain_to_layout(Ap.view(np.uint16), Bp.view(np.uint16), "m", "k")
    r = oracle.linear_forward(A, B, None, "none", M, N, K, a_major="m", b_major="k")
    ref = Ap.astype(np.float64) @ Bp.astype(np.float64)
    assert np.allclose(r["Z"].reshape(M, N), ref, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- DRELU

def test_drelu_bgrad_against_exact_sum(oracle):
    rng = np.random.default_rng(21)
    M, N, K = 45, 300, 16
    A = rng.standard_normal(M * K).astype(np.float16)
    B = rng.standard_normal(K * N).astype(np.float16)
    bias = rng.standard_normal(M).astype(np.float16)
    for dl in ("row", "col"):
        rows, cols = (M, N) if dl == "row" else (N, M)
        fw = oracle.linear_forward(A, B, bias, "relu_aux_bias", M, N, K, d_layout=dl)
        dY = (rng.standard_normal(rows * cols) * 3).astype(np.float16)
        dZ, bgrad = oracle.drelu_bgrad(dY, fw["aux"], M, N, d_layout=dl)
        mask = (fw["Z"] > 0)
        dYf = dY.astype(np.float64)
        ref_dz = np.where(mask, dYf, 0.0)
        assert np.array_equal(oracle.f16_decode(dZ), ref_dz)
        assert not (dZ[~mask] != 0).any()  # masked-out gradients are +0
        grid = ref_dz.reshape(rows, cols)
        per_m = grid if dl == "row" else grid.T
        for m in range(M):
            # a sum of fp16 values with this few terms is exact in fp64;
            # math.fsum (exact, reverse order) must agree to the last bit.
            assert bgrad[m] == math.fsum(per_m[m][::-1])


# ------------------------------------------------ DRELU_BGRAD on a product

def test_gemm_drelu_bgrad_hand_worked(oracle):
    """The hand-worked example's product A.B = [[0,13,3],[-2,5,1]] masked by
    [[1,1,1],[0,1,0]] gives dZ = [[0,13,3],[0,5,0]] and bgrad = [16, 5]."""
    g = json.load(open(os.path.join(GOLDEN, "hand_2x3x4.json")))
    M, N, K = g["M"], g["N"], g["K"]
    A = f16_bits(g["A"]).reshape(-1)
    B = f16_bits(g["B"]).reshape(-1)
    aux = np.array(g["mask_words_row_major_ld4"], np.uint32)
    dZ, bgrad = oracle.gemm_drelu_bgrad(A, B, aux, M, N, K, a_major="k", b_major="n", d_layout="row")
    assert oracle.f16_decode(dZ).reshape(M, N).tolist() == [[0, 13, 3], [0, 5, 0]]
    assert bgrad.tolist() == [16.0, 5.0]


@pytest.mark.parametrize("am,bm,dl", [("k", "n", "row"), ("k", "k", "col"), ("m", "n", "row"), ("m", "k", "col")])
def test_gemm_drelu_bgrad_brute_force(oracle, am, bm, dl):
    rng = np.random.default_rng(40 + "km".index(am) * 4 + "kn".index(bm) * 2 + (dl == "col"))
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (5, 33, 4), (37, 2, 9)]:
        Ap = rng.standard_normal((M, K)).astype(np.float16)
        Bp = rng.standard_normal((K, N)).astype(np.float16)
        rows, cols = (M, N) if dl == "row" else (N, M)
        ld_aux = 4 * ((cols + 127) // 128)
        bitmat = rng.integers(0, 2, (M, N))
        aux = np.zeros(rows * ld_aux, np.uint32)
        for m in range(M):
            for n in range(N):
                r, c = (m, n) if dl == "row" else (n, m)
                if bitmat[m, n]:
                    aux[r * ld_aux + c // 32] |= np.uint32(1 << (c % 32))
        A, B = plain_to_layout(Ap.view(np.uint16), Bp.view(np.uint16), am, bm)
        dZ, bgrad = oracle.gemm_drelu_bgrad(A, B, aux, M, N, K, a_major=am, b_major=bm, d_layout=dl, threads=1)
        Z, _ = _brute(Ap.astype(np.float64), Bp.astype(np.float64), None, "none")
        masked = np.where(bitmat == 1, Z, 0.0)
        want = np.where(bitmat == 1, Z, 0.0).astype(np.float16).view(np.uint16)
        got = dZ.reshape(rows, cols)
        if dl == "col":
            got = got.T
        assert np.array_equal(got, want)
        for m in range(M):
            s = 0.0
            for n in range(N):
                s += masked[m, n]
            assert bgrad[m] == s


# ------------------------------------------------------------- erf GELU

def test_gelu_erf_closed_forms(oracle):
    act = lambda z: oracle.act_f64("gelu_erf_bias", z)
    assert act(0.0) == 0.0
    assert abs(act(1.0) - 0.8413447460685429) < 1e-15  # Phi(1) = 0.841344746...
    assert act(12.0) == 12.0
    for z in np.linspace(-6, 6, 241):
        # z Phi(z) - (-z) Phi(-z) = z (Phi(z) + Phi(-z)) = z
        assert abs(act(z) - act(-z) - z) <= 4e-16 * max(1.0, abs(z))


def test_gelu_erf_matches_library(oracle):
    z = torch.linspace(-9, 9, 7001, dtype=torch.float64)
    ref = torch.nn.functional.gelu(z, approximate="none").numpy()
    got = np.array([oracle.act_f64("gelu_erf_bias", float(v)) for v in z])
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-15)
    # and it is not the tanh approximation
    tanh_form = np.array([oracle.act_f64("gelu_bias", float(v)) for v in z])
    assert np.abs(got - tanh_form).max() > 1e-5


def test_gelu_erf_forward_brute_force(oracle):
    rng = np.random.default_rng(77)
    M, N, K = 4, 5, 6
    Ap = rng.standard_normal((M, K)).astype(np.float16)
    Bp = rng.standard_normal((K, N)).astype(np.float16)
    bias = rng.standard_normal(M).astype(np.float16)
    A, B = plain_to_layout(Ap.view(np.uint16), Bp.view(np.uint16), "k", "n")
    r = oracle.linear_forward(A, B, bias.view(np.uint16), "gelu_erf_bias", M, N, K, a_major="k", b_major="n")
    Z = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += float(Ap[m, k]) * float(Bp[k, n])
            Z[m, n] = s + float(bias[m])
    want = torch.nn.functional.gelu(torch.from_numpy(Z), approximate="none").numpy()
    assert np.array_equal(r["D"].reshape(M, N), want.astype(np.float16).view(np.uint16))


# --------------------------------------------------------------- bfloat16

def test_bf16_decode_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_decode(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_encode_roundtrip_and_ties(oracle):
    bits = np.arange(0, 0x7F80, dtype=np.uint16)      # every finite positive bfloat16
    vals = oracle.bf16_decode(bits)
    assert np.array_equal(oracle.bf16_encode(vals), bits)
    assert np.array_equal(oracle.bf16_encode(-vals), bits | 0x8000)
    lo = bits[:-1]
    a, b = vals[:-1], vals[1:]
    mid = (a + b) / 2                                  # exact in fp64
    even = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(oracle.bf16_encode(mid), even)
    assert np.array_equal(oracle.bf16_encode(np.nextafter(mid, 0)), lo)
    assert np.array_equal(oracle.bf16_encode(np.nextafter(mid, np.inf)), (lo + 1).astype(np.uint16))


def test_bf16_encode_vs_library_on_float32_values(oracle):
    # For doubles that are exact float32 values, torch's float32 -> bfloat16
    # conversion (round to nearest even) is a single rounding: it must agree.
    rng = np.random.default_rng(9)
    x = (np.exp2(rng.uniform(-140, 127.9, 200000)) * rng.choice([-1.0, 1.0], 200000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_encode(x.astype(np.float64)), ref)


def test_bf16_encode_boundaries(oracle):
    enc = lambda v: int(oracle.bf16_encode(np.array([v]))[0])
    big = (2 - 2 ** -7) * 2.0 ** 127
    assert enc(big) == 0x7F7F
    assert enc((2 - 2 ** -8) * 2.0 ** 127) == 0x7F80   # tie to even -> overflow
    assert enc(2.0 ** -133) == 0x0001
    assert enc(2.0 ** -134) == 0x0000                 # tie to even -> zero
    assert enc(2.0 ** -126) == 0x0080


def test_bf16_forward_brute_force(oracle):
    rng = np.random.default_rng(78)
    M, N, K = 5, 4, 7
    tb = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    Ap = tb(rng.standard_normal((M, K)).astype(np.float32))
    Bp = tb(rng.standard_normal((K, N)).astype(np.float32))
    bias = tb(rng.standard_normal(M).astype(np.float32))
    bitsof = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
    r = oracle.linear_forward(bitsof(Ap), bitsof(Bp.T.contiguous()), bitsof(bias), "relu_bias", M, N, K,
                              a_major="k", b_major="k", dtype="bf16")
    Z = np.zeros((M, N))
    A64, B64, b64 = Ap.double().numpy(), Bp.double().numpy(), bias.double().numpy()
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += A64[m, k] * B64[k, n]
            Z[m, n] = max(s + b64[m], 0.0)
    want = torch.from_numpy(Z.astype(np.float32)).to(torch.bfloat16)  # Z is not exact in fp32:
    got = oracle.bf16_decode(r["D"]).reshape(M, N)
    # compare against round-to-nearest of the fp64 value instead (one rounding)
    assert np.array_equal(r["D"].reshape(M, N), oracle.bf16_encode(Z))
    assert np.allclose(got, want.double().numpy(), rtol=2 ** -7)


# ------------------------------------------- GELU_AUX_BIAS and DGELU_BGRAD

def _torch_gelu_grad(z):
    """d/dz of the library's tanh-form GELU, by autograd in fp64."""
    t = torch.tensor(np.asarray(z, np.float64), requires_grad=True)
    torch.nn.functional.gelu(t, approximate="tanh").sum().backward()
    return t.grad.numpy()


def test_gelu_grad_finite_difference(oracle):
    """The derivative matches a central difference of the (separately pinned)
    forward GELU: a wrong coefficient or a dropped chain-rule factor fails."""
    h = 1e-5
    for z in np.linspace(-8, 8, 401):
        fd = (oracle.act_f64("gelu_bias", z + h) - oracle.act_f64("gelu_bias", z - h)) / (2 * h)
        assert abs(oracle.gelu_grad_f64(z) - fd) < 1e-8, z


def test_gelu_grad_matches_library_autograd(oracle):
    z = np.linspace(-10, 10, 4001)
    got = np.array([oracle.gelu_grad_f64(v) for v in z])
    # For |z| > 7, 1 - t^2 is a few ulps of 1 in both evaluations, so their
    # absolute difference there is rounding noise of order 1e-15.
    assert np.allclose(got, _torch_gelu_grad(z), rtol=1e-13, atol=1e-14)


def test_gelu_grad_special_values(oracle):
    assert oracle.gelu_grad_f64(0.0) == 0.5
    assert abs(oracle.gelu_grad_f64(12.0) - 1.0) < 1e-15
    assert abs(oracle.gelu_grad_f64(-12.0)) < 1e-15
    # the derivative is negative for z below about -0.75 (minimum near -1.42)
    # and exceeds 1 for z above about 0.75
    assert oracle.gelu_grad_f64(-0.7) > 0 > oracle.gelu_grad_f64(-0.8)
    assert oracle.gelu_grad_f64(-1.5) < oracle.gelu_grad_f64(-1.2)
    assert oracle.gelu_grad_f64(-1.5) < oracle.gelu_grad_f64(-1.8)
    assert oracle.gelu_grad_f64(1.5) > 1


@pytest.mark.parametrize("dl", ["row", "col"])
def test_gelu_aux_forward(oracle, dl):
    """GELU_AUX_BIAS: D is the GELU_BIAS output and zaux is z = A.B + bias
    (brute force, fp64) rounded once to fp16 by the library conversion; the
    padding of each zaux row is left untouched."""
    rng = np.random.default_rng(90)
    M, N, K = 7, 11, 13
    Ap = rng.standard_normal((M, K)).astype(np.float16)
    Bp = rng.standard_normal((K, N)).astype(np.float16)
    bias = rng.standard_normal(M).astype(np.float16)
    A, B = plain_to_layout(Ap.view(np.uint16), Bp.view(np.uint16), "k", "n")
    rows, cols = (M, N) if dl == "row" else (N, M)
    r = oracle.linear_forward(A, B, bias.view(np.uint16), "gelu_aux_bias", M, N, K, a_major="k",
                              b_major="n", d_layout=dl)
    g = oracle.linear_forward(A, B, bias.view(np.uint16), "gelu_bias", M, N, K, a_major="k",
                              b_major="n", d_layout=dl)
    assert np.array_equal(r["D"], g["D"])
    ld = r["ld_zaux"]
    assert ld == (cols + 7) // 8 * 8
    Z = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += float(Ap[m, k]) * float(Bp[k, n])
            Z[m, n] = s + float(bias[m])
    want = Z if dl == "row" else Z.T
    zaux = r["zaux"].reshape(rows, ld)
    assert np.array_equal(zaux[:, :cols], want.astype(np.float16).view(np.uint16))
    assert not zaux[:, cols:].any()


@pytest.mark.parametrize("dl", ["row", "col"])
def test_dgelu_bgrad_standalone(oracle, dl):
    """dZ = dY * gelu'(z) rounded once; bgrad = sum over n of the unrounded
    products. gelu' comes from the library's autograd here."""
    rng = np.random.default_rng(91)
    M, N = 9, 40
    rows, cols = (M, N) if dl == "row" else (N, M)
    ldd, ldz = cols + 3, cols + 5
    dY = (rng.standard_normal((rows, ldd)) * 2).astype(np.float16)
    z = (rng.standard_normal((rows, ldz)) * 3).astype(np.float16)
    dZ, bgrad = oracle.dgelu_bgrad(dY.view(np.uint16).reshape(-1), z.view(np.uint16).reshape(-1), M, N,
                                   d_layout=dl, ldd=ldd, ld_zaux=ldz)
    g = dY[:, :cols].astype(np.float64) * _torch_gelu_grad(z[:, :cols].astype(np.float64))
    got = dZ.reshape(rows, ldd)
    assert np.array_equal(got[:, :cols], g.astype(np.float16).view(np.uint16))
    assert not got[:, cols:].any()  # padding untouched
    per_m = g if dl == "row" else g.T
    assert np.allclose(bgrad, [math.fsum(per_m[m]) for m in range(M)], rtol=1e-13, atol=1e-13)


def test_dgelu_bgrad_special_values(oracle):
    """gelu'(0) = 1/2 (exact halving), gelu'(8) rounds to 1 (dZ = dY) and
    gelu'(-8) is below 1e-19 in magnitude (dZ is a zero)."""
    dY = np.array([1.5, -3.0, 2.0], np.float16)
    z = np.array([0.0, 8.0, -8.0], np.float16)
    dZ, bgrad = oracle.dgelu_bgrad(dY.view(np.uint16), z.view(np.uint16), 1, 3)
    assert dZ[:2].tolist() == [np.float16(0.75).view(np.uint16), np.float16(-3.0).view(np.uint16)]
    assert dZ[2] & 0x7FFF == 0
    assert abs(bgrad[0] - (0.75 - 3.0)) < 1e-15


@pytest.mark.parametrize("am,bm,dl", [("k", "n", "row"), ("k", "k", "col"), ("m", "n", "row"), ("m", "k", "col")])
def test_gemm_dgelu_bgrad_brute_force(oracle, am, bm, dl):
    rng = np.random.default_rng(92 + "km".index(am) * 4 + "kn".index(bm) * 2 + (dl == "col"))
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (6, 33, 4)]:
        Ap = rng.standard_normal((M, K)).astype(np.float16)
        Bp = rng.standard_normal((K, N)).astype(np.float16)
        rows, cols = (M, N) if dl == "row" else (N, M)
        ldz = (cols + 7) // 8 * 8
        zs = (rng.standard_normal((rows, ldz)) * 2).astype(np.float16)
        A, B = plain_to_layout(Ap.view(np.uint16), Bp.view(np.uint16), am, bm)
        dZ, bgrad = oracle.gemm_dgelu_bgrad(A, B, zs.view(np.uint16).reshape(-1), M, N, K, a_major=am,
                                            b_major=bm, d_layout=dl, threads=1)
        H, _ = _brute(Ap.astype(np.float64), Bp.astype(np.float64), None, "none")
        zmn = zs[:, :cols].astype(np.float64)
        if dl == "col":
            zmn = zmn.T
        g = H * _torch_gelu_grad(zmn)
        got = dZ.reshape(rows, cols)
        if dl == "col":
            got = got.T
        assert np.array_equal(got, g.astype(np.float16).view(np.uint16))
        assert np.allclose(bgrad, g.sum(axis=1), rtol=1e-13, atol=1e-14)


def test_dgelu_bgrad_bf16(oracle):
    """bf16 elements: the same products rounded by the (separately pinned)
    bf16 encoder."""
    rng = np.random.default_rng(93)
    tb = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    bitsof = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
    M, N = 6, 17
    dY = tb(rng.standard_normal((M, N)) * 2)
    z = tb(rng.standard_normal((M, N)) * 3)
    ldz = (N + 7) // 8 * 8
    zp = torch.zeros((M, ldz), dtype=torch.bfloat16)
    zp[:, :N] = z
    dZ, bgrad = oracle.dgelu_bgrad(bitsof(dY), bitsof(zp), M, N, ld_zaux=ldz, dtype="bf16")
    g = dY.double().numpy() * _torch_gelu_grad(z.double().numpy())
    assert np.array_equal(dZ.reshape(M, N), oracle.bf16_encode(g))
    assert np.allclose(bgrad, g.sum(axis=1), rtol=1e-13, atol=1e-14)


# ------------------------------- MatMul + bias + residual + RMSNorm / LayerNorm

def _norm_inputs(rng, M, N, K, dtype=np.float16):
    A = rng.standard_normal((M, K)).astype(dtype)
    B = rng.standard_normal((K, N)).astype(dtype)
    bias = rng.standard_normal(M).astype(dtype)
    res = rng.standard_normal((M, N)).astype(dtype)
    gamma = (1 + 0.5 * rng.standard_normal(M)).astype(dtype)
    beta = rng.standard_normal(M).astype(dtype)
    return A, B, bias, res, gamma, beta


def _run_norm(oracle, A, B, bias, res, gamma, beta, norm, eps, dl="col"):
    """A [M,K], B [K,N], res [M,N] plain fp16 arrays; returns H, Y as [M,N] fp64."""
    M, K = A.shape
    N = B.shape[1]
    Ak, Bk = plain_to_layout(A.view(np.uint16), B.view(np.uint16), "k", "n")
    r = res if dl == "row" else res.T
    H, Y = oracle.linear_norm(Ak, Bk, bias.view(np.uint16), np.ascontiguousarray(r).view(np.uint16).reshape(-1),
                              gamma.view(np.uint16), None if beta is None else beta.view(np.uint16), norm, M, N, K,
                              eps=eps, a_major="k", b_major="n", d_layout=dl)
    rows, cols = (M, N) if dl == "row" else (N, M)
    H = oracle.f16_decode(H).reshape(rows, cols)
    Y = oracle.f16_decode(Y).reshape(rows, cols)
    return (H, Y) if dl == "row" else (H.T, Y.T)


def test_layernorm_two_features_is_plus_minus_one(oracle):
    """Over two features LayerNorm gives +-sqrt(v/(v+eps)) (v = the variance):
    exactly +1 / -1 with eps = 0, for the hand-worked example's z."""
    g = json.load(open(os.path.join(GOLDEN, "hand_2x3x4.json")))
    A = np.array(g["A"], np.float16)
    B = np.array(g["B"], np.float16)
    bias = np.array(g["bias"], np.float16)
    zeros = np.zeros((2, 3), np.float16)
    one = np.ones(2, np.float16)
    H, Y = _run_norm(oracle, A, B, bias, zeros, one, np.zeros(2, np.float16), "layernorm", 0.0)
    assert H.tolist() == [[0.5, 13.5, 3.5], [-5, 2, -2]]
    assert Y.tolist() == [[1, 1, 1], [-1, -1, -1]]
    # eps > 0: token 0 has h = (0.5, -5), variance 2.75^2
    _, Y = _run_norm(oracle, A, B, bias, zeros, one, np.zeros(2, np.float16), "layernorm", 1.0)
    want = np.sqrt(2.75 ** 2 / (2.75 ** 2 + 1.0))
    assert Y[0, 0] == np.float16(want) and Y[1, 0] == np.float16(-want)


def test_rmsnorm_closed_forms(oracle):
    """h = (3, 4): rms = sqrt(12.5), so y = (3, 4) * sqrt(2) / 5; a constant
    row c gives sign(c) * gamma (eps = 0)."""
    A = np.array([[3.0], [4.0]], np.float16)
    B = np.array([[1.0, -2.0]], np.float16)
    z2 = np.zeros(2, np.float16)
    _, Y = _run_norm(oracle, A, B, z2, np.zeros((2, 2), np.float16), np.ones(2, np.float16), None, "rmsnorm", 0.0)
    s2 = 1.4142135623730951
    assert Y[:, 0].tolist() == [float(np.float16(3 * s2 / 5)), float(np.float16(4 * s2 / 5))]
    assert Y[:, 1].tolist() == [float(np.float16(-3 * s2 / 5)), float(np.float16(-4 * s2 / 5))]
    M = 7
    A = np.full((M, 1), 0.75, np.float16)
    gamma = np.linspace(-2, 2, M).astype(np.float16)
    _, Y = _run_norm(oracle, A, np.array([[1.0, -3.0]], np.float16), np.zeros(M, np.float16),
                     np.zeros((M, 2), np.float16), gamma, None, "rmsnorm", 0.0)
    assert np.array_equal(Y[:, 0], gamma.astype(np.float64))
    assert np.array_equal(Y[:, 1], -gamma.astype(np.float64))


def test_norm_scale_invariance(oracle):
    """With eps = 0 both norms ignore a common scale of h: doubling A, the
    bias and the residual (exact in fp16) doubles H and leaves Y unchanged."""
    rng = np.random.default_rng(95)
    A, B, bias, res, gamma, beta = _norm_inputs(rng, 24, 5, 9)
    for norm in ("rmsnorm", "layernorm"):
        H1, Y1 = _run_norm(oracle, A, B, bias, res, gamma, beta, norm, 0.0)
        H2, Y2 = _run_norm(oracle, A * np.float16(2), B, bias * np.float16(2), res * np.float16(2), gamma, beta,
                           norm, 0.0)
        assert np.array_equal(H2, 2 * H1)
        assert np.array_equal(Y1, Y2)


def test_layernorm_output_moments(oracle):
    """gamma = 1, beta = 0: each token's outputs have mean 0 and variance
    v / (v + eps) up to the fp16 rounding of Y."""
    rng = np.random.default_rng(96)
    M, N, K = 256, 6, 16
    A, B, bias, res, _, _ = _norm_inputs(rng, M, N, K)
    eps = 0.5
    H, Y = _run_norm(oracle, A, B, bias, res, np.ones(M, np.float16), np.zeros(M, np.float16), "layernorm", eps)
    h = A.astype(np.float64) @ B.astype(np.float64) + bias.astype(np.float64)[:, None] + res.astype(np.float64)
    v = h.var(axis=0)
    assert np.abs(Y.mean(axis=0)).max() < 2e-3
    assert np.abs(Y.var(axis=0) - v / (v + eps)).max() < 4e-3


@pytest.mark.parametrize("norm", ["rmsnorm", "layernorm"])
@pytest.mark.parametrize("dl", ["row", "col"])
def test_norm_brute_force(oracle, norm, dl):
    """Brute force on tiny inputs: h by explicit loops, the statistics by
    numpy's mean and (population) variance, one rounding by the library."""
    rng = np.random.default_rng(97 + (norm == "layernorm") * 2 + (dl == "col"))
    for (M, N, K) in [(1, 1, 1), (5, 3, 7), (33, 4, 5)]:
        A, B, bias, res, gamma, beta = _norm_inputs(rng, M, N, K)
        H, Y = _run_norm(oracle, A, B, bias, res, gamma, beta if norm == "layernorm" else None, norm, 1e-5, dl)
        h = np.zeros((M, N))
        for m in range(M):
            for n in range(N):
                s = 0.0
                for k in range(K):
                    s += float(A[m, k]) * float(B[k, n])
                h[m, n] = s + float(bias[m]) + float(res[m, n])
        assert np.array_equal(H, h.astype(np.float16).astype(np.float64))
        if norm == "rmsnorm":
            y = h / np.sqrt((h * h).mean(axis=0) + 1e-5) * gamma.astype(np.float64)[:, None]
        else:
            y = (h - h.mean(axis=0)) / np.sqrt(h.var(axis=0) + 1e-5) * gamma.astype(np.float64)[:, None] \
                + beta.astype(np.float64)[:, None]
        # Y is y rounded once: within half an fp16 step of the brute-force y
        half_step = np.spacing(np.abs(y).astype(np.float16)).astype(np.float64) / 2
        assert (np.abs(Y - y) <= half_step * (1 + 1e-9) + 1e-300).all(), "Y differs from the brute force"


@pytest.mark.parametrize("norm", ["rmsnorm", "layernorm"])
def test_norm_matches_library_norms(oracle, norm):
    """Against torch's own LayerNorm / RMSNorm in fp64 over each token's M
    features (h from the library matmul): Y is their result rounded once."""
    import torch.nn.functional as F
    rng = np.random.default_rng(98 + (norm == "layernorm"))
    M, N, K = 96, 7, 24
    A, B, bias, res, gamma, beta = _norm_inputs(rng, M, N, K)
    eps = 1e-5
    H, Y = _run_norm(oracle, A, B, bias, res, gamma, beta if norm == "layernorm" else None, norm, eps)
    h = torch.from_numpy(A.astype(np.float64)) @ torch.from_numpy(B.astype(np.float64)) \
        + torch.from_numpy(bias.astype(np.float64))[:, None] + torch.from_numpy(res.astype(np.float64))
    g = torch.from_numpy(gamma.astype(np.float64))
    if norm == "layernorm":
        y = F.layer_norm(h.T, (M,), g, torch.from_numpy(beta.astype(np.float64)), eps).T
    else:
        y = F.rms_norm(h.T, (M,), g, eps).T
    y = y.numpy()
    half_step = np.spacing(np.abs(y).astype(np.float16)).astype(np.float64) / 2
    assert (np.abs(Y - y) <= half_step * (1 + 1e-6)).all(), "Y differs from the library norm"


def test_norm_bf16(oracle):
    rng = np.random.default_rng(99)
    M, N, K = 16, 3, 5
    tb = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)
    bitsof = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
    A, B = tb(rng.standard_normal((M, K))), tb(rng.standard_normal((K, N)))
    bias, res = tb(rng.standard_normal(M)), tb(rng.standard_normal((N, M)))
    gamma, beta = tb(1 + 0.3 * rng.standard_normal(M)), tb(rng.standard_normal(M))
    H, Y = oracle.linear_norm(bitsof(A), bitsof(B.T), bitsof(bias), bitsof(res), bitsof(gamma), bitsof(beta),
                              "layernorm", M, N, K, eps=1e-5, a_major="k", b_major="k", d_layout="col",
                              dtype="bf16")
    h = A.double().numpy() @ B.double().numpy() + bias.double().numpy()[:, None] + res.double().numpy().T
    y = (h - h.mean(axis=0)) / np.sqrt(h.var(axis=0) + 1e-5) * gamma.double().numpy()[:, None] \
        + beta.double().numpy()[:, None]
    assert np.array_equal(H.reshape(N, M), oracle.bf16_encode(h.T))
    got = oracle.bf16_decode(Y).reshape(N, M)
    assert np.abs(got - y.T).max() <= np.abs(y).max() * 2 ** -8


def test_dw_drelu_bgrad_brute_force(oracle):
    """Weight gradient with the ReLU backward on its A operand: brute force
    from an explicit bit array (dZ = dY where the bit is set, dW = dZ^T X,
    bgrad = column sums of dZ over the tokens), padded pitches."""
    rng = np.random.default_rng(97)
    for (M, N, K) in [(1, 1, 1), (5, 3, 7), (40, 9, 33)]:
        lda, ldx = M + 3, N + 2
        ld_aux = (M + 127) // 128 * 4
        dY = rng.standard_normal((K, lda)).astype(np.float16)
        X = rng.standard_normal((K, ldx)).astype(np.float16)
        keep = rng.random((K, M)) < 0.6
        words = np.zeros((K, ld_aux), np.uint32)
        for k in range(K):
            for m in range(M):
                if keep[k, m]:
                    words[k, m // 32] |= np.uint32(1 << (m % 32))
        dW, bgrad = oracle.dw_drelu_bgrad(dY.view(np.uint16).reshape(-1), words.reshape(-1),
                                          X.view(np.uint16).reshape(-1), M, N, K, lda=lda, ldb=ldx,
                                          ld_aux=ld_aux)
        dZ = np.where(keep, dY[:, :M].astype(np.float64), 0.0)
        want = np.zeros((M, N))
        for m in range(M):
            for n in range(N):
                want[m, n] = math.fsum(dZ[k, m] * float(X[k, n]) for k in range(K))
        assert np.array_equal(dW.reshape(M, N), want.astype(np.float16).view(np.uint16))
        assert np.allclose(bgrad, [math.fsum(dZ[:, m]) for m in range(M)], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- decode chain
def _f16_bits(x):
    return np.asarray(x, np.float16).view(np.uint16).reshape(-1)


def test_decode_chain_permutation_then_its_transpose_is_identity(oracle):
    """W0 = P (a permutation, not symmetric), W1 = P^T: layer 0 permutes the
    token's features, layer 1 undoes it, exactly. A transposed weight, a
    swapped layer order or a lost intermediate would fail."""
    M, N = 7, 2
    perm = np.array([3, 0, 6, 1, 5, 2, 4])
    P = np.zeros((M, M))
    P[np.arange(M), perm] = 1.0  # (P x)[i] = x[perm[i]]
    X = np.arange(N * M, dtype=np.float64).reshape(N, M) - 5.0
    y0, y1 = oracle.decode_chain([_f16_bits(P), _f16_bits(P.T)], [None, None], _f16_bits(X), "none", M, N)
    assert np.array_equal(oracle.f16_decode(y0).reshape(N, M), X[:, perm])
    assert np.array_equal(y1, _f16_bits(X))


def test_decode_chain_bias_accumulates_through_identity_layers(oracle):
    """W = I with a BIAS epilogue: Y_l = X + b_0 + ... + b_l (small integers,
    exact in fp16)."""
    M, N, L = 9, 3, 4
    I = _f16_bits(np.eye(M))
    rng = np.random.default_rng(5)
    X = rng.integers(-4, 5, (N, M)).astype(np.float64)
    bs = [rng.integers(-3, 4, M).astype(np.float64) for _ in range(L)]
    outs = oracle.decode_chain([I] * L, [_f16_bits(b) for b in bs], _f16_bits(X), "bias", M, N)
    acc = X.copy()
    for l in range(L):
        acc = acc + bs[l][None, :]
        assert np.array_equal(oracle.f16_decode(outs[l]).reshape(N, M), acc)


def test_decode_chain_relu_closed_form(oracle):
    """W = I, bias -1, ReLU: Y_l = max(X - (l + 1), 0)."""
    M, N, L = 6, 2, 3
    X = np.array([[0, 1, 2, 3, 4, -2], [5, 6, -1, 2, 0, 9]], np.float64)
    outs = oracle.decode_chain([_f16_bits(np.eye(M))] * L, [_f16_bits(-np.ones(M))] * L, _f16_bits(X),
                               "relu_bias", M, N)
    for l in range(L):
        assert np.array_equal(oracle.f16_decode(outs[l]).reshape(N, M), np.maximum(X - (l + 1), 0))


def test_decode_chain_matches_numpy_layer_by_layer(oracle):
    """Random chain with tanh-GELU against an independent numpy computation:
    fp64 product and bias, the tanh form of GELU, then numpy's own round to
    nearest even fp16 before the next layer."""
    M, N, L = 24, 2, 3
    rng = np.random.default_rng(11)
    Ws = [rng.standard_normal((M, M)).astype(np.float16) / np.float16(4) for _ in range(L)]
    bs = [(rng.standard_normal(M) * 0.3).astype(np.float16) for _ in range(L)]
    X = rng.standard_normal((N, M)).astype(np.float16)
    outs = oracle.decode_chain([w.view(np.uint16).reshape(-1) for w in Ws],
                               [b.view(np.uint16) for b in bs], X.view(np.uint16).reshape(-1),
                               "gelu_bias", M, N)
    x = X.astype(np.float64)
    for l in range(L):
        z = x @ Ws[l].astype(np.float64).T + bs[l].astype(np.float64)[None, :]
        y = 0.5 * z * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (z + 0.044715 * z ** 3)))
        y16 = y.astype(np.float16)
        assert np.array_equal(outs[l], y16.view(np.uint16).reshape(-1)), f"layer {l}"
        x = y16.astype(np.float64)
