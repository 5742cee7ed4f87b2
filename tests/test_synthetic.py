"""The seeded input generator: rounding and workload bookkeeping (CPU)."""
import numpy as np
import pytest

from exact_attention_41_gb300 import synthetic as syn


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(100_000).astype(np.float32) * 7
    x[:4] = [1.00390625, 1.01171875, -2.0039062, 3.0e-39]  # ties and a subnormal
    bits = syn.round_bits(x, syn.BF16)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, want)
    np.testing.assert_array_equal(syn.bits_to_f64(bits, syn.BF16),
                                  torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_f16_rounding_round_trips():
    x = np.random.default_rng(1).standard_normal(1000).astype(np.float32)
    bits = syn.round_bits(x, syn.F16)
    np.testing.assert_array_equal(syn.bits_to_f64(bits, syn.F16), x.astype(np.float16).astype(np.float64))


def test_varlen_lengths_and_cu_seqlens():
    lens = syn.varlen_lengths(7)
    assert len(lens) == 64 and lens.min() >= 100 and lens.max() <= 4096
    cu = syn.cu_seqlens(lens)
    assert cu.dtype == np.int32 and cu[0] == 0 and (np.diff(cu) == lens).all()
    assert syn.cu_seqlens([100, 200, 150]).tolist() == [0, 100, 300, 450]


def test_decode_layout_is_a_permutation():
    seqlens, table, n = syn.decode_layout(8, 64, 32768, 256, 4)
    assert table.shape == (64, 129) and n == 8256
    assert sorted(table.ravel().tolist()) == list(range(n))
    assert seqlens.min() >= 1 and seqlens.max() <= 32768
    assert ((seqlens + 4) <= 129 * 256).all()


def test_same_seed_same_bits():
    a = syn.dense_case(3, 1, 8, 8, 2, 1, 16, syn.BF16, with_dout=True)
    b = syn.dense_case(3, 1, 8, 8, 2, 1, 16, syn.BF16, with_dout=True)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])
