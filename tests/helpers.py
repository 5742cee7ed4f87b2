"""Shared test utilities: moving seeded bits to the device and back, and the
tolerance contract.

Tolerances (elementwise, against the float64 oracle):
  fp16: |gpu - ref| <= 2e-3 + 2e-3 * |ref|
  bf16: |gpu - ref| <= 1e-2 + 1e-2 * |ref|
  LSE (fp32): |gpu - ref| <= 1e-3, and -inf exactly where the oracle has -inf.
The FlashAttention FAQ's own reference tolerances (Inference Cookbook Q10:
fp16 1e-3/1e-3, bf16 5e-3/5e-3) are tighter; `report` records how a result
fares against both, without asserting, and the test session prints the
table at its end (tests/conftest.py).
"""
import numpy as np

from exact_attention_41_gb300 import synthetic as syn

TOL = {syn.F16: (2e-3, 2e-3), syn.BF16: (1e-2, 1e-2)}
PAGE_TOL = {syn.F16: (1e-3, 1e-3), syn.BF16: (5e-3, 5e-3)}
LSE_TOL = 1e-3


def dev(bits, dtype):
    """uint16 bits -> CUDA tensor of the storage dtype (same bits)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.float16 if dtype == syn.F16 else torch.bfloat16)


def dev_i32(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host(t):
    """Device tensor -> float64 numpy (exact widening)."""
    import torch

    return t.detach().to(torch.float64).cpu().numpy()


def f64(bits, dtype):
    return syn.bits_to_f64(bits, dtype)


def assert_close(got, want, dtype, what=""):
    atol, rtol = TOL[dtype]
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance "
            f"(worst at {idx}: got {got[idx]}, want {want[idx]}); max abs err {err.max():.3e}")


def assert_lse(got, want, what="lse"):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    ninf = np.isneginf(want)
    assert (np.isneginf(got) == ninf).all(), f"{what}: -inf pattern differs"
    err = np.abs(got[~ninf] - want[~ninf])
    assert err.size == 0 or err.max() <= LSE_TOL, f"{what}: max abs err {err.max():.3e}"


def max_err(got, want):
    return float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))))


# (name, reference, dtype, max |err|, worst err/bound and fraction out of
# bound for the contract, the same for the FAQ's tolerances)
ACCURACY = []


def error_stats(got, want, dtype):
    """Max |err| and, for the contract and the FAQ Q10 tolerances, the worst
    err / bound ratio and the fraction of elements above the bound."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    out = {"max_abs_err": float(err.max()) if err.size else 0.0}
    for name, (atol, rtol) in (("contract", TOL[dtype]), ("pages_q10", PAGE_TOL[dtype])):
        bound = atol + rtol * np.abs(want)
        out[name] = {"worst_ratio": float((err / bound).max()) if err.size else 0.0,
                     "frac_out": float((err > bound).mean()) if err.size else 0.0}
    return out


def report(name, got, want, dtype, reference="oracle (stored-O reading of D)"):
    """Records how `got` compares with `want` against both tolerance sets;
    asserts nothing."""
    ACCURACY.append((name, reference, dtype, error_stats(got, want, dtype)))
