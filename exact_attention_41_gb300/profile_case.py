"""Runs one attention kernel on a small, fixed case, for profiler captures.

    python -m exact_attention_41_gb300.profile_case fwd     # b=1 s=8192 hq=16 hkv=4 d=128 causal
    python -m exact_attention_41_gb300.profile_case bwd
    python -m exact_attention_41_gb300.profile_case decode  # b=8 sq=4, caches U[1,32768]

Each runs `--calls` calls (default 2: one warm-up, one to capture) and checks
the device error word.  Inputs are seeded N(0,1) bf16 drawn on the device;
the problems are larger than L2 in their K/V or Q/dO streams and at most
about 1 GB in total.
"""
from __future__ import annotations

import argparse
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def main():
    import torch

    from exact_attention_41_gb300 import libattn
    from exact_attention_41_gb300 import synthetic as syn

    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["fwd", "bwd", "decode"])
    ap.add_argument("--calls", type=int, default=2)
    ap.add_argument("--b", type=int, default=1)
    ap.add_argument("--s", type=int, default=8192)
    ap.add_argument("--hq", type=int, default=16)
    ap.add_argument("--hkv", type=int, default=4)
    ap.add_argument("--deterministic", action="store_true")
    args = ap.parse_args()
    bf = syn.BF16
    d = 128
    if args.kernel in ("fwd", "bwd"):
        q = syn.device_normal((args.b, args.s, args.hq, d), bf, 1)
        k = syn.device_normal((args.b, args.s, args.hkv, d), bf, 2)
        v = syn.device_normal((args.b, args.s, args.hkv, d), bf, 3)
        if args.kernel == "fwd":
            for _ in range(args.calls):
                libattn.fwd(q, k, v, causal=True)
        else:
            do = syn.device_normal((args.b, args.s, args.hq, d), bf, 4)
            o, lse = libattn.fwd(q, k, v, causal=True)
            for _ in range(args.calls):
                libattn.bwd(q, k, v, o, lse, do, causal=True, deterministic=args.deterministic)
    else:
        b, sq, page = 8, 4, 256
        seqlens, table, npages = syn.decode_layout(9, b, 32768, page, sq)
        kc = syn.device_normal((npages, page, args.hkv * 2, d), bf, 5)
        vc = syn.device_normal((npages, page, args.hkv * 2, d), bf, 6)
        q = syn.device_normal((b, sq, args.hkv * 8, d), bf, 7)
        kn = syn.device_normal((b, sq, args.hkv * 2, d), bf, 8)
        vn = syn.device_normal((b, sq, args.hkv * 2, d), bf, 9)
        sl = torch.from_numpy(seqlens).cuda()
        bt = torch.from_numpy(table).cuda()
        for _ in range(args.calls):
            libattn.fwd_kvcache(q, kc, vc, sl, k_new=kn, v_new=vn, block_table=bt, causal=True)
    torch.cuda.synchronize()
    st = libattn.device_error()
    print("done", args.kernel, "device error", st)
    sys.exit(0 if st == (0, 0) else 1)


if __name__ == "__main__":
    main()
