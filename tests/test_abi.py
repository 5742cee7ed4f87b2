"""The C ABI on the host: the library loads, exports every declared symbol,
and rejects invalid calls before touching a device (no GPU needed)."""
import ctypes

import pytest

from exact_attention_41_gb300 import build as build_mod
from exact_attention_41_gb300 import libattn


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return libattn.lib()


def test_exports_every_declared_function(lib):
    names = libattn.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(libattn._SIGS), "binding signatures out of sync with the header"


def test_version_and_status_strings(lib):
    assert lib.attn_version().startswith(b"libattn")
    assert lib.attn_status_str(0) == b"ok"
    assert lib.attn_status_str(3) == b"workspace missing or too small"


def test_workspace_sizes(lib):
    # D (b*hq*sq fp32) + dQ accumulator (b*sq*hq*d fp32) + counters
    n = lib.attn_bwd_workspace_size(4, 8192, 8192, 32, 8, 128, 0)
    assert n >= 4 * 8192 * 32 * 4 * (1 + 128)
    assert lib.attn_bwd_workspace_size(0, 8, 8, 1, 1, 64, 0) == 0
    assert lib.attn_kvcache_workspace_size(64, 1, 32, 8, 128, 33024, 1) == 0
    s = lib.attn_kvcache_num_splits(64, 1, 32, 8, 128, 33024, 5)
    assert s == 5
    assert lib.attn_kvcache_workspace_size(64, 1, 32, 8, 128, 33024, 5) >= 5 * 64 * 32 * 128 * 4


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


def fwd(lib, **over):
    a = dict(dtype=1, b=1, sq=8, sk=8, hq=4, hkv=2, d=128, scale=0.1, causal=0, wl=-1, wr=-1,
             cap=0.0)
    a.update(over)
    return lib.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, a["dtype"], a["b"], a["sq"], a["sk"],
                        a["hq"], a["hkv"], a["d"], a["scale"], a["causal"], a["wl"], a["wr"],
                        a["cap"], None)


@pytest.mark.parametrize("over,status", [
    (dict(d=96), 2), (dict(d=32), 2), (dict(hq=6, hkv=4), 1), (dict(hkv=0), 1),
    (dict(dtype=7), 1), (dict(wl=-2), 1), (dict(wr=-5), 1), (dict(scale=float("inf")), 1),
    (dict(scale=-0.5), 1), (dict(scale=float("nan")), 1),
    (dict(cap=float("nan")), 1), (dict(b=-1), 1), (dict(sq=-3), 1),
])
def test_invalid_arguments_are_rejected_on_host(lib, over, status):
    assert fwd(lib, **over) == status


def test_empty_problem_is_a_noop(lib):
    assert fwd(lib, b=0) == 0
    assert fwd(lib, sq=0) == 0


def test_misaligned_pointer_rejected(lib):
    bad = ctypes.c_void_p(0x10002)
    st = lib.attn_fwd(bad, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 8, 4, 2, 128, 0.1, 0, -1, -1, 0.0,
                      None)
    assert st == 1


def test_bwd_workspace_checked(lib):
    st = lib.attn_bwd(*([FAKE] * 9), 1, 1, 8, 8, 4, 2, 128, 0.1, 0, -1, -1, 0.0, 0, FAKE, 16,
                      None)
    assert st == 3


def test_kvcache_argument_checks(lib):
    args = lambda **o: dict(dict(num_pages=4, page_size=256, maxp=2, b=2, sq=1, s_new=1, bt=FAKE), **o)

    def call(a):
        return lib.attn_fwd_kvcache(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["bt"], a["num_pages"],
                                    a["page_size"], a["maxp"], FAKE, FAKE, 1, a["b"], a["sq"],
                                    a["s_new"], 32, 8, 128, 0.1, 1, -1, -1, 0.0, 0, FAKE, 1 << 30,
                                    None)

    assert call(args(page_size=100)) == 1          # pages must be a multiple of 128
    assert call(args(bt=None, num_pages=4)) == 1   # contiguous: one page per entry
    assert call(args(s_new=-1)) == 1
    assert call(args(b=0)) == 0


def test_probs_and_advance_argument_checks(lib):
    probs = lambda p=FAKE, b=1, hq=4, hkv=2, d=128: lib.attn_fwd_probs(
        FAKE, FAKE, FAKE, p, 1, b, 8, 8, hq, hkv, d, 0.1, 0, -1, -1, 0.0, None)
    assert probs(hq=6, hkv=4) == 1       # hq not a multiple of hkv
    assert probs(d=96) == 2              # head dim not supported
    assert probs(p=None) == 1            # no output
    assert probs(b=0) == 0               # empty problem: no-op
    assert lib.attn_kvcache_advance(FAKE, -1, 1, None) == 1
    assert lib.attn_kvcache_advance(FAKE, 2, -1, None) == 1
    assert lib.attn_kvcache_advance(None, 2, 1, None) == 1
    assert lib.attn_kvcache_advance(ctypes.c_void_p(0x10002), 2, 1, None) == 1  # misaligned
    assert lib.attn_kvcache_advance(FAKE, 0, 1, None) == 0


def test_strided_argument_checks(lib):
    def fwd_s(qs=0, ks=0, vs=0):
        return lib.attn_fwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, qs, ks, vs, 1, 1, 8, 8, 4, 2,
                                    128, 0.1, 0, -1, -1, 0.0, -1, None)
    assert fwd_s(qs=4 * 128 - 8) == 1     # a token row shorter than its heads
    assert fwd_s(ks=2 * 128 + 4) == 1     # not a multiple of 8 elements
    assert fwd_s(vs=-8) == 1
    bwd_s = lambda dk: lib.attn_bwd_strided(*([FAKE] * 9), 0, 0, 0, 0, dk, 0, 1, 1, 8, 8, 4, 2,
                                            128, 0.1, 0, -1, -1, 0.0, 0, FAKE, 1 << 30, None)
    assert bwd_s(2 * 128 - 8) == 1
    assert lib.attn_fwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, 3 * 4 * 128, 0, 0, 1, 0, 8, 8, 4, 2,
                                128, 0.1, 0, -1, -1, 0.0, -1, None) == 0   # empty: no-op
    # PackGQA forced on needs hq / hkv to divide the 128-row tile
    assert lib.attn_fwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 0, 1, 1, 8, 8, 6, 2,
                                128, 0.1, 0, -1, -1, 0.0, 1, None) == 2


def test_fp8_host_checks(lib):
    call = lambda dq=1.0, d=128, sk=8, ws=1 << 30: lib.attn_fwd_fp8(
        FAKE, FAKE, FAKE, FAKE, FAKE, dq, 1.0, 1.0, 1, 8, sk, 4, 2, d, 0.1, 0, -1, -1, 0.0, FAKE,
        ws, None)
    assert call(dq=0.0) == 1 and call(dq=float("inf")) == 1
    assert call(d=64) == 2 and call(sk=0) == 2
    assert call(ws=16) == 3
    assert lib.attn_fwd_fp8_workspace_size(2, 100, 8, 128) >= 2 * 100 * 8 * 128 * 2


def test_split_heuristic_on_host(lib):
    """Inference Cookbook FAQ Q14's split rules as implemented (host logic;
    the SM count is the present GPU's, 152 -- the GB300's -- without one):
    enough (batch, KV head) units and short caches -> one split; long caches
    -> 8192-key pieces; few units -> at least SMs / units splits, never more
    than 128-key tiles; an explicit request wins."""
    sms = 152
    if libattn_has_device():
        import torch

        sms = torch.cuda.get_device_properties(0).multi_processor_count
    ns = lambda b, hkv, cap, n=0: lib.attn_kvcache_num_splits(b, 1, 32, hkv, 128, cap, n)
    assert ns(64, 8, 4096) == (1 if 64 * 8 >= sms else -(-sms // 512))
    assert ns(64, 8, 33024) == max(5, -(-sms // 512))
    assert ns(1, 8, 4096) == min(-(-sms // 8), 32)   # ceil(SMs / units), <= 32 tiles
    assert ns(1, 8, 1000) == 8                       # capped by the 8 key tiles
    assert ns(64, 8, 33024, 3) == 3


def libattn_has_device():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False
