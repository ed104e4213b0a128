"""Pins for the oracle's block-scaled fp8 dispatch payload.

The pages say dispatch carries tokens with block scaling factors
("Efficient and portable mixture-of-experts communication", Dispatch) and that
the evaluated kernels use block-scale fp8 dispatch with bf16 combine
("Enabling trillion-parameter models on AWS EFA", evaluation); they do not
give the block size or the scale rule.  The oracle reads them as blocks of
128 consecutive elements, E4M3 codes, scale = amax / 448, inv = 1 / scale
(both float32 divisions, once per block) and q = round-to-nearest-even(x * inv).
Pins:

* the E4M3 rounding against torch's float32 -> float8_e4m3fn conversion (a
  library routine) inside the finite range, and the decoding of all 256 codes;
* saturation above the largest finite value (448) and signed zeros;
* a hand-worked block; the largest element maps to +-448 exactly; an all-zero
  block has scale 1 and zero codes; the dequantised values stay within half an
  E4M3 step of the inputs.
"""
import numpy as np
import pytest
import torch

from combine_route_count_gb300 import inputs as gen


def torch_e4m3(vals):
    t = torch.tensor(np.asarray(vals, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_rounding_matches_torch(oracle_mod):
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.uniform(-460, 460, 3000),
        rng.standard_normal(3000) * 10,
        rng.standard_normal(1000) * 1e-2,   # subnormal range of E4M3 (< 2^-6)
        np.array([0.0, 1.0, -1.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 0.015625]),
        # exact ties between neighbouring codes: 1 + 1/16 lies between 1 and 1.125
        np.array([1.0625, 1.1875, 17.0, 19.0, 240.0, 272.0]),
    ]).astype(np.float32)
    want = torch_e4m3(vals)
    got = np.array([oracle_mod.float_to_e4m3(float(v)) for v in vals], np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_decoding_of_every_code(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = np.array([oracle_mod.e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # every finite code survives a round trip
    for c in codes[~nan]:
        assert oracle_mod.float_to_e4m3(float(oracle_mod.e4m3_to_double(int(c)))) == int(c)


def test_e4m3_saturates_at_448(oracle_mod):
    for v in (448.0, 449.0, 463.9, 464.0, 1e6, 3.0e38):
        assert oracle_mod.float_to_e4m3(v) == 0x7E
        assert oracle_mod.float_to_e4m3(-v) == 0xFE
    assert oracle_mod.float_to_e4m3(-0.0) == 0x80
    assert oracle_mod.float_to_e4m3(0.0) == 0x00


def test_hand_worked_block(oracle_mod):
    """Block [1, 2, -3, 0, 0, ...]: amax 3, scale 3/448, inv = 1/scale ~ 149.33;
    1*inv = 149.33 -> nearest E4M3 144 = 1.125 * 2^7 -> code 0x71;
    2*inv = 298.67 -> nearest 288 = 1.125 * 2^8 -> code 0x79;
    -3*inv = -448 (within rounding) -> code 0xFE; zeros -> 0x00."""
    x = np.zeros((1, 128), np.float32)
    x[0, :3] = [1.0, 2.0, -3.0]
    q, sc = oracle_mod.quantize_fp8(gen.to_bf16_bits(x))
    assert sc[0, 0] == np.float32(3.0) / np.float32(448.0)
    assert q[0, :4].tolist() == [0x71, 0x79, 0xFE, 0x00]
    assert np.all(q[0, 4:] == 0)


def test_quantisation_properties(oracle_mod):
    rng = np.random.default_rng(12)
    T, H = 24, 7168
    xf = rng.standard_normal((T, H)).astype(np.float32) * np.exp(rng.uniform(-6, 6, (T, 1))).astype(np.float32)
    xf[3, 128:256] = 0.0  # an all-zero block
    x = gen.to_bf16_bits(xf)
    q, sc = oracle_mod.quantize_fp8(x)
    assert q.shape == (T, H) and sc.shape == (T, H // 128)
    xv = gen.bf16_bits_to_f32(x).reshape(T, H // 128, 128).astype(np.float64)
    amax = np.abs(xv).max(axis=2)
    nz = amax > 0
    assert np.array_equal(sc[nz], (amax[nz].astype(np.float32) / np.float32(448.0)))
    assert sc[3, 1] == 1.0 and np.all(q[3, 128:256] == 0)
    # the largest element of each non-zero block maps to +-448
    qb = q.reshape(T, H // 128, 128)
    arg = np.abs(xv).argmax(axis=2)
    top = np.take_along_axis(qb, arg[..., None], axis=2)[..., 0]
    assert np.all((top[nz] & 0x7F) == 0x7E)
    # dequantised values within half an E4M3 step of x (relative 2^-4 for
    # normal codes, absolute 2^-10 * scale in the subnormal range)
    deq = np.vectorize(oracle_mod.e4m3_to_double)(qb) * sc[..., None].astype(np.float64)
    err = np.abs(deq - xv)
    bound = np.maximum(np.abs(xv) * 2.0 ** -4, sc[..., None].astype(np.float64) * 2.0 ** -10) * 1.0001
    assert np.all(err <= bound)


def test_fp8_dispatch_places_the_quantised_rows(oracle_mod):
    w = gen.custom("fp8", T=64, H=256, K=4, E=16, N=4, seed_index=13)
    li = gen.make_inputs(w, with_y=False)
    d, xq, xs = oracle_mod.dispatch_fp8(li.x, li.topk_idx, w.E, w.N)
    q, sc = oracle_mod.quantize_fp8(li.x)
    for row in range(w.T * w.K):
        t = d.row_src[row] // w.K
        assert np.array_equal(xq[row], q[t]) and np.array_equal(xs[row], sc[t])


def test_fp8_rejects_rows_not_a_multiple_of_the_block(oracle_mod):
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.quantize_fp8(np.zeros((2, 200), np.uint16))
