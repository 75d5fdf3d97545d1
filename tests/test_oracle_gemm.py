"""Pins of the oracle's grouped fp8 GEMM (the expert stand-in that consumes
the block-scaled dispatch layout of "Efficient and portable mixture-of-experts
communication", §Dispatch).

Independent ground truth only: e4m3 decoding by PyTorch's float8_e4m3fn,
float64 matrix products by numpy, closed forms whose results are exactly
representable in bf16, and hand-built rounding ties.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def bf16_values(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def bf16_bits_exact(v: np.ndarray) -> np.ndarray:
    """bf16 bits of values that are exactly representable (asserted)."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float64))
    b = t.to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(b.to(torch.float64).numpy(), v), "value not representable in bf16"
    return b.view(torch.int16).numpy().view(np.uint16)


def random_codes(rng, shape):
    """Any finite e4m3 code (zeros, subnormals, both signs, up to 448); no NaN."""
    c = rng.integers(0, 254, size=shape, dtype=np.int64)
    c = np.where(c >= 0x7F, c + 1, c)          # skip 0x7F
    return c.astype(np.uint8)                    # 0x80..0xFE (0xFF never drawn)


def reference(q, sa, w, sw):
    """float64 value of the definition, blockwise, with numpy matmul."""
    E, C, K = q.shape
    N = w.shape[1]
    qa, wa = e4m3_values(q), e4m3_values(w)
    out = np.zeros((E, C, N))
    for b in range(K // 128):
        blk = np.einsum("eck,enk->ecn", qa[:, :, b * 128:(b + 1) * 128], wa[:, :, b * 128:(b + 1) * 128])
        wsc = np.repeat(sw[:, :, b].astype(np.float64), 128, axis=1)          # [E][N]
        out += blk * sa[:, :, b].astype(np.float64)[:, :, None] * wsc[:, None, :]
    return out


def assert_nearest_bf16(y_bits, exact):
    """y is a nearest bf16 to the exact value (half an ulp of the bf16 grid at y)."""
    y = bf16_values(y_bits)
    a = np.abs(y)
    ex = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    ulp = np.where(a > 0, 2.0 ** (ex - 7), 2.0 ** -133)
    assert np.all(np.abs(y - exact) <= 0.5 * ulp * (1 + 1e-12)), np.max(np.abs(y - exact) / ulp)


@pytest.mark.parametrize("K,N", [(256, 384), (384, 128), (128, 128)])
def test_gemm_equals_float64_matmul(K, N):
    rng = np.random.default_rng(K + N)
    E, C = 3, 5
    q = random_codes(rng, (E, C, K))
    sa = rng.uniform(0.01, 2.0, size=(E, C, K // 128)).astype(np.float32)
    w = random_codes(rng, (E, N, K))
    sw = rng.uniform(0.001, 0.1, size=(E, N // 128, K // 128)).astype(np.float32)
    counts = np.array([5, 2, 0], dtype=np.int32)
    y = O.expert_gemm_fp8(q, sa, counts, w, sw)
    ref = reference(q, sa, w, sw)
    for e in range(E):
        r = min(int(counts[e]), C)
        assert_nearest_bf16(y[e, :r], ref[e, :r])
        assert not y[e, r:].any(), "rows past the count must stay untouched"


def test_identity_weights_give_the_dequantised_rows():
    """W = I, weight scales 1: y = q * a_scale, exact in bf16 when the scale is a power of two."""
    rng = np.random.default_rng(5)
    E, C, K = 2, 4, 256
    q = random_codes(rng, (E, C, K))
    sa = (2.0 ** rng.integers(-6, 6, size=(E, C, K // 128))).astype(np.float32)
    w = np.zeros((E, K, K), dtype=np.uint8)
    w[:, np.arange(K), np.arange(K)] = 0x38                                  # 1.0
    sw = np.ones((E, K // 128, K // 128), dtype=np.float32)
    y = O.expert_gemm_fp8(q, sa, np.array([C, C], dtype=np.int32), w, sw)
    want = e4m3_values(q) * np.repeat(sa.astype(np.float64), 128, axis=2) + 0.0    # sums start at +0
    assert np.array_equal(y, bf16_bits_exact(want))


def test_permutation_weights_pick_inputs_and_block_scales():
    """W[n][pi(n)] = 1 with pi crossing 128-blocks and not an involution, weight
    block scales 2^(3*nb + kb): y[r][n] = q[r][pi(n)] * a_scale[r][pi(n)/128]
    * 2^(3*(n/128) + pi(n)/128). A transposed W or a wrong scale index fails."""
    rng = np.random.default_rng(6)
    E, C, K = 1, 3, 384
    pi = rng.permutation(K)
    assert not np.array_equal(pi[pi], np.arange(K))
    q = random_codes(rng, (E, C, K))
    sa = (2.0 ** rng.integers(-4, 4, size=(E, C, K // 128))).astype(np.float32)
    w = np.zeros((E, K, K), dtype=np.uint8)
    w[0, np.arange(K), pi] = 0x38
    nb, kb = np.meshgrid(np.arange(K // 128), np.arange(K // 128), indexing="ij")
    sw = (2.0 ** (3 * nb + kb)).astype(np.float32)[None]
    y = O.expert_gemm_fp8(q, sa, np.array([C], dtype=np.int32), w, sw)
    n = np.arange(K)
    want = (e4m3_values(q[0][:, pi]) * sa[0][:, pi // 128].astype(np.float64)
            * (2.0 ** (3 * (n // 128) + pi // 128))[None, :]) + 0.0
    assert np.array_equal(y[0], bf16_bits_exact(want))


def test_rounding_is_once_to_nearest_even():
    """1 + 2^-8 is a tie between bf16 1.0 and 1 + 2^-7: even wins (1.0).
    1 + 2^-7 + 2^-8 ties between 1 + 2^-7 and 1 + 2^-6: even wins (1 + 2^-6).
    1 + 2^-8 + 2^-40 is above the tie: it must round up, which a detour through
    float32 (where 2^-40 is lost) would miss."""
    K, N = 256, 128
    q = np.zeros((1, 3, K), dtype=np.uint8)
    q[0, :, 0] = 0x38                 # 1.0
    q[0, 0, 1] = 0x02                 # 2^-8 (subnormal: 2/8 * 2^-6)
    q[0, 1, 1] = 0x02
    q[0, 1, 2] = 0x04                 # 2^-7
    q[0, 2, 1] = 0x02
    q[0, 2, 128] = 0x38               # second block: 1.0, scaled by 2^-40 below
    sa = np.ones((1, 3, 2), dtype=np.float32)
    sa[0, 2, 1] = 2.0 ** -40
    w = np.zeros((1, N, K), dtype=np.uint8)
    w[0, 0, :3] = 0x38
    w[0, 0, 128] = 0x38
    sw = np.ones((1, 1, 2), dtype=np.float32)
    y = O.expert_gemm_fp8(q, sa, np.array([3], dtype=np.int32), w, sw)
    assert [hex(v) for v in y[0, :, 0]] == ["0x3f80", "0x3f82", "0x3f81"]
    assert not y[0, :, 1:].any()


def test_capacity_clips_rows_and_row_entry_matches():
    w_ = W.Workload("g", T=0, H=256, E=2, k=1, R=1, C=4, dtype=1, seed=77)
    rng = np.random.default_rng(8)
    q = random_codes(rng, (2, 4, 256))
    sa = rng.uniform(0.5, 1.5, size=(2, 4, 2)).astype(np.float32)
    wq, ws = W.make_weights(w_)
    y = O.expert_gemm_fp8(q, sa, np.array([9, 1], dtype=np.int32), wq, ws)
    assert y[0].any(axis=1).all() and not y[1, 1:].any()
    for e, r in [(0, 0), (0, 3), (1, 0)]:
        assert np.array_equal(O.gemm_fp8_row(q[e, r], sa[e, r], wq[e], ws[e]), y[e, r])


def test_weight_generator_draws_the_stated_distribution():
    w_ = W.WORKLOADS["tiny"]
    wq, ws = W.make_weights(w_)
    mag = wq & 0x7F
    assert mag.min() == 0x30 and mag.max() == 0x77
    v = np.abs(e4m3_values(wq))
    assert v.min() == 0.5 and v.max() == 240.0
    assert 0.45 < (wq >> 7).mean() < 0.55
    assert ws.min() >= 2.0 ** -8 and ws.max() < 2.0 ** -7
    a, b = W.make_weights(w_, e0=5, ne=2)
    assert np.array_equal(a, wq[5:7]) and np.array_equal(b, ws[5:7])


# ---- bf16 rows, bf16 weights --------------------------------------------------

def random_bf16(rng, shape, scale=1.0):
    return torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("K,N", [(256, 384), (72, 40), (1, 3)])
def test_bf16_gemm_equals_float64_matmul(K, N):
    rng = np.random.default_rng(K * 7 + N)
    E, C = 3, 4
    x = random_bf16(rng, (E, C, K))
    w = random_bf16(rng, (E, N, K), 2.0 ** -5)
    counts = np.array([4, 1, 0], dtype=np.int32)
    y = O.expert_gemm_bf16(x, counts, w)
    ref = np.einsum("eck,enk->ecn", bf16_values(x), bf16_values(w))
    for e in range(E):
        r = min(int(counts[e]), C)
        assert_nearest_bf16(y[e, :r], ref[e, :r])
        assert not y[e, r:].any()


def test_bf16_identity_and_permutation_weights_are_exact():
    """W = I gives the rows back (zeros as +0); a permutation that is not an
    involution, with power-of-two weights 2^(n mod 5), gives x[pi(n)] * 2^(n mod 5):
    a transposed W fails."""
    rng = np.random.default_rng(11)
    K = 96
    x = random_bf16(rng, (1, 3, K))
    eye = np.zeros((1, K, K), dtype=np.uint16)
    eye[0, np.arange(K), np.arange(K)] = 0x3F80
    y = O.expert_gemm_bf16(x, np.array([3], dtype=np.int32), eye)
    assert np.array_equal(y, bf16_bits_exact(bf16_values(x) + 0.0))
    pi = rng.permutation(K)
    assert not np.array_equal(pi[pi], np.arange(K))
    n = np.arange(K)
    wp = np.zeros((1, K, K), dtype=np.uint16)
    wp[0, n, pi] = bf16_bits_exact((2.0 ** (n % 5)).astype(np.float64))
    y = O.expert_gemm_bf16(x, np.array([3], dtype=np.int32), wp)
    want = bf16_values(x[0][:, pi]) * (2.0 ** (n % 5))[None, :] + 0.0
    assert np.array_equal(y[0], bf16_bits_exact(want))


def test_bf16_rounding_is_once_to_nearest_even():
    """1 + 2^-8 ties to 1.0; 1 + 2^-8 + 2^-40 must round up to 1 + 2^-7."""
    x = np.zeros((1, 2, 3), dtype=np.uint16)
    x[0, 0, :2] = [0x3F80, 0x3B80]            # 1, 2^-8
    x[0, 1, :] = [0x3F80, 0x3B80, 0x2B80]     # 1, 2^-8, 2^-40
    w = np.full((1, 1, 3), 0x3F80, dtype=np.uint16)
    y = O.expert_gemm_bf16(x, np.array([2], dtype=np.int32), w)
    assert [hex(v) for v in y[0, :, 0]] == ["0x3f80", "0x3f81"]


def test_bf16_weight_generator_and_row_entry():
    w_ = W.WORKLOADS["tiny"]
    wb = W.make_weights_bf16(w_)
    v = bf16_values(wb)
    assert wb.shape == (8, 256, 256) and abs(v.std() - 2.0 ** -5) < 2.0 ** -9 and abs(v.mean()) < 2.0 ** -10
    assert np.array_equal(W.make_weights_bf16(w_, e0=3, ne=2), wb[3:5])
    rng = np.random.default_rng(3)
    x = random_bf16(rng, (8, 4, 256))
    y = O.expert_gemm_bf16(x, np.full(8, 4, dtype=np.int32), wb)
    assert np.array_equal(O.gemm_bf16_row(x[5, 2], wb[5]), y[5, 2])
