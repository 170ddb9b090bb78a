"""Pins for the CPU oracle, against facts fixed by arithmetic, by the pages'
definition of C = A x B, and by independent library routines (numpy BLAS,
torch dtype conversion).  None of these calls the oracle twice and compares it
with itself; each would fail on a dropped term, a wrong sign or index, or a
transposed operand."""

import numpy as np
import pytest
import torch

from dense_int8_matrix_gb300 import workloads


def _np_i8(t):
    return t.numpy() if isinstance(t, torch.Tensor) else t


def _bits(t_bf16: torch.Tensor) -> np.ndarray:
    return t_bf16.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- int8 ----

def test_all_int8_pairs_brute_force(oracle_mod):
    # k = 1: C[i][j] = a_i * b_j for every one of the 256 x 256 value pairs,
    # including (-128)*(-128) = 16384 and (-128)*127 = -16256.
    vals = np.arange(-128, 128, dtype=np.int64)
    A = vals.astype(np.int8).reshape(256, 1)
    Bt = vals.astype(np.int8).reshape(256, 1)
    C = oracle_mod.gemm_i8(A, Bt)
    expect = np.array([[a * b for b in range(-128, 128)] for a in range(-128, 128)])
    assert np.array_equal(C.astype(np.int64), expect)
    assert C[0, 0] == 16384 and C[0, 255] == -16256 and C[255, 255] == 16129


@pytest.mark.parametrize("m,k,n,seed", [(37, 129, 53, 1), (1, 1000, 7, 2),
                                        (64, 4096, 3, 3), (130, 65, 260, 4)])
def test_matches_numpy_int64_matmul(oracle_mod, m, k, n, seed):
    A = _np_i8(workloads.random_i8((m, k), seed))
    Bt = _np_i8(workloads.random_i8((n, k), seed + 100))
    C = oracle_mod.gemm_i8(A, Bt, nthreads=3)
    ref = A.astype(np.int64) @ Bt.astype(np.int64).T
    assert C.dtype == np.int32
    assert np.array_equal(C.astype(np.int64), ref)


def test_all_ones_gives_k(oracle_mod):
    m, k, n = 17, 333, 29
    C = oracle_mod.gemm_i8(np.ones((m, k), np.int8), np.ones((n, k), np.int8))
    assert np.all(C == k)


def test_identity_gives_b(oracle_mod):
    k, n = 48, 21
    Bt = _np_i8(workloads.random_i8((n, k), 7))
    C = oracle_mod.gemm_i8(np.eye(k, dtype=np.int8), Bt)
    # A = I: C[i][j] = B[i][j] = Bt[j][i]
    assert np.array_equal(C, Bt.T.astype(np.int32))


def test_transpose_identity(oracle_mod):
    # (A B)^T = B^T A^T: swapping the roles of A and Bt transposes C.
    A = _np_i8(workloads.random_i8((23, 70), 8))
    Bt = _np_i8(workloads.random_i8((31, 70), 9))
    C = oracle_mod.gemm_i8(A, Bt)
    Ct = oracle_mod.gemm_i8(Bt, A)
    assert np.array_equal(Ct, C.T)


def test_zero_row_gives_zero_row(oracle_mod):
    A = _np_i8(workloads.random_i8((9, 40), 10)).copy()
    A[4] = 0
    Bt = _np_i8(workloads.random_i8((12, 40), 11))
    C = oracle_mod.gemm_i8(A, Bt)
    assert np.all(C[4] == 0) and np.any(C[3] != 0)


def test_extreme_magnitude_k16384(oracle_mod):
    k = 16384
    A = np.full((2, k), -128, np.int8)
    Bt = np.full((3, k), -128, np.int8)
    C = oracle_mod.gemm_i8(A, Bt)
    assert np.all(C == 16384 * k) and C[0, 0] == 2 ** 28


def test_overflow_is_reported_not_wrapped(oracle_mod):
    k_ok = 131071          # 131071 * 16384 = 2^31 - 16384 fits int32
    C = oracle_mod.gemm_i8(np.full((1, k_ok), -128, np.int8),
                           np.full((1, k_ok), -128, np.int8))
    assert C[0, 0] == 131071 * 16384
    k_bad = 131073         # 2^31 + 16384 does not
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.gemm_i8(np.full((1, k_bad), -128, np.int8),
                           np.full((1, k_bad), -128, np.int8))


def test_freivalds_property(oracle_mod):
    # C r == A (B r) exactly in int64, for random integer vectors r.
    m, k, n = 96, 512, 80
    A = _np_i8(workloads.random_i8((m, k), 12))
    Bt = _np_i8(workloads.random_i8((n, k), 13))
    C = oracle_mod.gemm_i8(A, Bt).astype(np.int64)
    rng = np.random.default_rng(5)
    for _ in range(3):
        r = rng.integers(-1000, 1000, size=n, dtype=np.int64)
        br = Bt.astype(np.int64).T @ r
        assert np.array_equal(C @ r, A.astype(np.int64) @ br)


def test_entries_match_full(oracle_mod):
    A = _np_i8(workloads.random_i8((50, 300), 14))
    Bt = _np_i8(workloads.random_i8((40, 300), 15))
    rows = np.array([0, 49, 17, 3, 49])
    cols = np.array([0, 39, 5, 38, 0])
    got = oracle_mod.gemm_i8_entries(A, Bt, rows, cols)
    ref = A.astype(np.int64)[rows] * Bt.astype(np.int64)[cols]
    assert np.array_equal(got, ref.sum(axis=1))


def test_empty_shapes(oracle_mod):
    C = oracle_mod.gemm_i8(np.zeros((0, 5), np.int8), np.zeros((3, 5), np.int8))
    assert C.shape == (0, 3)
    C = oracle_mod.gemm_i8(np.zeros((4, 0), np.int8), np.zeros((3, 0), np.int8))
    assert C.shape == (4, 3) and np.all(C == 0)


# ---------------------------------------------------------------- bf16 ----

def test_bf16_widening_all_bit_patterns(oracle_mod):
    # C = a * 1.0 must reproduce every bf16 value as torch widens it.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(-1, 1)
    one = np.array([[0x3F80]], dtype=np.uint16)
    C, S = oracle_mod.gemm_bf16(bits, one)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert np.array_equal(C, ref, equal_nan=True)
    finite = np.isfinite(ref[:, 0])
    assert np.array_equal(S[finite, 0], np.abs(ref[finite, 0]).astype(np.float64))


def test_bf16_known_products(oracle_mod):
    # 1.5 * 3.0 + (-2.0) * 0.25 = 4.0 ; S = 4.5 + 0.5
    A = np.array([[0x3FC0, 0xC000]], dtype=np.uint16)
    Bt = np.array([[0x4040, 0x3E80]], dtype=np.uint16)
    C, S = oracle_mod.gemm_bf16(A, Bt)
    assert C[0, 0] == np.float32(4.0) and S[0, 0] == 5.0


def test_bf16_integer_inputs_equal_int_oracle(oracle_mod):
    # |x| <= 16 is exact in bf16 and every partial sum stays far below 2^24,
    # so the bf16 product must equal the exact integer product.
    m, k, n = 33, 700, 45
    Ai = _np_i8(workloads.random_i8((m, k), 16, -16, 16))
    Bi = _np_i8(workloads.random_i8((n, k), 17, -16, 16))
    Ab = _bits(torch.from_numpy(Ai.astype(np.float32)).to(torch.bfloat16))
    Bb = _bits(torch.from_numpy(Bi.astype(np.float32)).to(torch.bfloat16))
    C, S = oracle_mod.gemm_bf16(Ab, Bb)
    Ci = oracle_mod.gemm_i8(Ai, Bi)
    assert np.array_equal(C, Ci.astype(np.float32))
    assert np.array_equal(S, np.abs(Ai.astype(np.int64)) @ np.abs(Bi.astype(np.int64)).T)


@pytest.mark.parametrize("m,k,n", [(19, 257, 23), (64, 1024, 8)])
def test_bf16_matches_numpy_float64(oracle_mod, m, k, n):
    A = workloads.random_bf16((m, k), 18)
    Bt = workloads.random_bf16((n, k), 19)
    C, S = oracle_mod.gemm_bf16(_bits(A), _bits(Bt))
    A64 = A.double().numpy()
    B64 = Bt.double().numpy()
    ref = A64 @ B64.T
    ref_abs = np.abs(A64) @ np.abs(B64).T
    # two double sums in different orders differ by ~k * 2^-53 * S; after one
    # rounding to float they agree to within one float ulp of the result
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(C.astype(np.float64) - ref) <= ulp + 1e-12 * ref_abs)
    assert np.allclose(S, ref_abs, rtol=1e-12, atol=0)


def test_bf16_entries_match_full(oracle_mod):
    A = workloads.random_bf16((20, 130), 20)
    Bt = workloads.random_bf16((15, 130), 21)
    C, S = oracle_mod.gemm_bf16(_bits(A), _bits(Bt))
    rows = np.array([0, 19, 7])
    cols = np.array([14, 0, 7])
    s, sa = oracle_mod.gemm_bf16_entries(_bits(A), _bits(Bt), rows, cols)
    assert np.array_equal(s.astype(np.float32), C[rows, cols])
    assert np.array_equal(sa, S[rows, cols])


# ------------------------------------------------------------ workloads ----

def test_workload_generators_shapes_and_ranges():
    A, Bt = workloads.make_inputs("i8_skinny", (8, 256, 512))
    assert A.shape == (8, 256) and Bt.shape == (512, 256)
    assert int(A.min()) >= -64 and int(A.max()) <= 63
    assert int(Bt.min()) >= -128 and int(Bt.max()) <= 127
    A2, Bt2 = workloads.make_inputs("i8_skinny", (8, 256, 512))
    assert torch.equal(A, A2) and torch.equal(Bt, Bt2)
    A3, _ = workloads.make_inputs("i8_skinny", (8, 256, 512), seed_offset=1)
    assert not torch.equal(A, A3)
    A, Bt = workloads.make_inputs("bf16_8192", (4, 64, 8))
    assert A.dtype == torch.bfloat16 and Bt.shape == (8, 64)


# ---------------------------------------------------------- requantisation ----
# D = q((float(C) * row_scale[i]) * col_scale[j]); the expected values below
# are worked out by hand from the binary32 and bfloat16 formats.

def _rq(oracle_mod, C, rs, cs, out):
    C = np.asarray(C, np.int32).reshape(len(rs), len(cs))
    return oracle_mod.requant(C, np.asarray(rs, np.float32), np.asarray(cs, np.float32), out)


def test_requant_int8_rounds_half_to_even_and_saturates(oracle_mod):
    # C * 0.5: 2.5 -> 2, 3.5 -> 4, -2.5 -> -2, -3.5 -> -4, 0.5 -> 0, 1.5 -> 2,
    # -1.5 -> -2, 9.5 -> 10, -8.5 -> -8; 255.5 rounds to 256 and saturates to
    # 127, -257 saturates to -128
    C = [5, 7, -5, -7, 1, 3, -3, 19, -17, 511, -514]
    got = _rq(oracle_mod, C, [0.5], [1.0] * 11, "i8")
    want = [2, 4, -2, -4, 0, 2, -2, 10, -8, 127, -128]
    assert got.tolist() == [want]


def test_requant_bf16_ties_to_even(oracle_mod):
    # 257 lies halfway between the bfloat16 values 256 (0x4380) and 258
    # (0x4381): the even one, 256; 259 halfway between 258 and 260 (0x4382):
    # 260; small integers are exact: 1 = 0x3f80, -2 = 0xc000, 3 = 0x4040
    got = _rq(oracle_mod, [257, 259, -257, 1, -2, 3], [1.0], [1.0] * 6, "bf16")
    assert got.tolist() == [[0x4380, 0x4382, 0xC380, 0x3F80, 0xC000, 0x4040]]


def test_requant_rounds_c_to_float_first(oracle_mod):
    # 16842753 = 2^24 + 2^16 + 1 is not a float: step (1) rounds it to
    # 2^24 + 2^16 (even), which is halfway between the bfloat16 values 2^24
    # (0x4b80) and 2^24 + 2^17 (0x4b81), so bfloat16 rounding gives 0x4b80.
    # Rounding the integer straight to bfloat16 would give 0x4b81.
    got = _rq(oracle_mod, [16842753], [1.0], [1.0], "bf16")
    assert got.tolist() == [[0x4B80]]


def test_requant_order_row_scale_then_column_scale(oracle_mod):
    # C = 2^30, row scale 2^100, column scale 2^-100: step (2) overflows to
    # infinity, which step (3) keeps (bfloat16 0x7f80, int8 saturates to 127).
    # Multiplying the two scales first would give exactly 2^30 (0x4e80).
    rs, cs = [2.0 ** 100], [2.0 ** -100]
    assert _rq(oracle_mod, [2 ** 30], rs, cs, "bf16").tolist() == [[0x7F80]]
    assert _rq(oracle_mod, [2 ** 30], rs, cs, "i8").tolist() == [[127]]
    # and infinity times a zero column scale is NaN: int8 0, bfloat16 NaN
    assert _rq(oracle_mod, [2 ** 30], rs, [0.0], "i8").tolist() == [[0]]
    nan = _rq(oracle_mod, [2 ** 30], rs, [0.0], "bf16")[0, 0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0


def test_requant_unit_scales_reproduce_small_integers(oracle_mod):
    vals = np.arange(-128, 128, dtype=np.int32)
    got = _rq(oracle_mod, vals, [1.0], [1.0] * 256, "i8")
    assert np.array_equal(got[0].astype(np.int32), vals)


def test_requant_rounding_matches_torch_on_arbitrary_floats(oracle_mod):
    # with C = 1 and column scale 1, steps (1)-(3) return the row scale x
    # unchanged, so D = q(x): compare q with torch's own float -> bfloat16
    # conversion and with torch.round (ties to even) + clamp, on random
    # finite binary32 bit patterns and on exact bfloat16 ties
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ties = (rng.integers(0, 2 ** 16, size=4000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    small = (rng.standard_normal(5000) * 200).astype(np.float32)
    halves = (np.arange(-300, 300, dtype=np.float32) + np.float32(0.5))
    x = np.concatenate([x, ties, small, halves]).astype(np.float32)
    C = np.ones((x.size, 1), np.int32)
    d16 = oracle_mod.requant(C, x, np.ones(1, np.float32), "bf16")[:, 0]
    ref16 = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(d16, ref16)
    d8 = oracle_mod.requant(C, x, np.ones(1, np.float32), "i8")[:, 0]
    ref8 = torch.round(torch.from_numpy(x).double()).clamp(-128, 127).to(torch.int8).numpy()
    assert np.array_equal(d8, ref8)


def test_requant_row_and_column_scales_index_the_right_axis(oracle_mod):
    # a 2 x 3 case by hand: C = [[10, 20, 30], [-40, 50, -60]],
    # row scales [0.5, 0.25], column scales [1, 2, 0.1]
    # row 0: 10*.5*1 = 5, 20*.5*2 = 20, 30*.5 = 15, and 15 times the float
    #        0.1 (0.100000001490116) is 1.50000002235, which rounds to the
    #        float 1.5 (spacing 2^-23 there), a tie that rounds to 2
    # row 1: -40*.25 = -10, 50*.25*2 = 25, -60*.25 = -15 -> -1.5 -> -2
    C = [[10, 20, 30], [-40, 50, -60]]
    got = _rq(oracle_mod, C, [0.5, 0.25], [1.0, 2.0, 0.1], "i8")
    assert got.tolist() == [[5, 20, 2], [-10, 25, -2]]
    # the transposed roles give a different answer, so a swapped index fails
    assert got.tolist() != _rq(oracle_mod, C, [1.0, 2.0], [0.5, 0.25, 1.0], "i8").tolist()
