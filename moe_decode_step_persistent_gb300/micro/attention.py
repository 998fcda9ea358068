"""Attention alone, through the allocation-free entry point
(msk_attention_noalloc: split-KV attention and the combine, the same phase
code the layer kernel runs): the full workload's head shape (16 verify
tokens, 32 query heads, 8 KV heads, head dim 128) over 16,384 cached tokens,
global and with a 2048-token window.  The 67 MB KV cache stays in L2 between
calls, so the times show the SM side of the phase, not HBM.

  python -m moe_decode_step_persistent_gb300.micro.attention            # times, one JSON line per case
  python -m moe_decode_step_persistent_gb300.micro.attention --profile  # 3 global calls, untimed (for ncu)
"""

from __future__ import annotations

import argparse
import json
import sys

import torch

T, HQ, HKV, D, S = 16, 32, 8, 128, 16384


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--profile", action="store_true", help="three untimed global calls and exit")
    p.add_argument("--calls", type=int, default=20)
    args = p.parse_args(argv)
    import moe_decode_step_persistent_gb300 as M
    M.load_library()
    g = torch.Generator(device="cuda").manual_seed(0)
    q = torch.randn((T, HQ, D), device="cuda", generator=g).to(torch.bfloat16)
    kv = torch.randn((2, HKV, S + 64, D), device="cuda", generator=g).to(torch.bfloat16)
    out = torch.empty((T, HQ * D), dtype=torch.bfloat16, device="cuda")
    for window in ((0,) if args.profile else (0, 2048)):
        for _ in range(3):
            if M.msk_attention_noalloc(q, kv, S, window, out) != M.MSK_OK:
                raise RuntimeError("msk_attention_noalloc failed")
        torch.cuda.synchronize()
        if args.profile:
            continue
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for _ in range(args.calls):
            M.msk_attention_noalloc(q, kv, S, window, out)
        ev[1].record()
        torch.cuda.synchronize()
        us = ev[0].elapsed_time(ev[1]) / args.calls * 1e3
        print(json.dumps({"probe": "attention_alone", "window": window, "cached": S, "tokens": T,
                          "q_heads": HQ, "kv_heads": HKV, "head_dim": D, "us_per_call": round(us, 1),
                          "kv_in_l2": True}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
