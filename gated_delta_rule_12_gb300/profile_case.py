"""Run one entry point a few times on seeded synthetic inputs, for a profiler to capture.

    python -m gated_delta_rule_12_gb300.profile_case --op bwd --B 2 --L 2048 --H 16 --calls 3

Each call goes through the C ABI on the current CUDA device, exactly as a user makes it; nothing
is timed or checked here. The inputs follow the library's input recipe (q, k, v Gaussian and
rounded to the element type; g = -0.1 softplus(z); beta = sigmoid(z)), so a capture sees the same
kernels and launch shapes as the timed runs, on a size chosen to keep the capture small.
"""
import argparse

import torch

import gated_delta_rule_12_gb300 as gdn
from gated_delta_rule_12_gb300 import inputs


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--op", choices=["fwd", "bwd", "decode", "decode_multi"], required=True)
    ap.add_argument("--B", type=int, default=1, help="sequences (decode: N)")
    ap.add_argument("--L", type=int, default=2048, help="tokens per sequence (decode_multi: tokens per call)")
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--dk", type=int, default=128)
    ap.add_argument("--dv", type=int, default=128)
    ap.add_argument("--dtype", choices=["bf16", "f32"], default="bf16")
    ap.add_argument("--calls", type=int, default=3)
    a = ap.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("profile_case needs a CUDA device")
    dev = torch.device("cuda", torch.cuda.current_device())
    gdn.load_library()
    elem = torch.bfloat16 if a.dtype == "bf16" else torch.float32

    if a.op in ("fwd", "bwd"):
        d = inputs.make_prefill(a.B, a.L, a.H, a.dk, a.dv, a.dtype, seed=1, init_state=True)
        d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in d.items()}
        if a.op == "fwd":
            for _ in range(a.calls):
                gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], init_state=d["init_state"])
        else:
            gen = torch.Generator().manual_seed(2)
            dO = torch.randn((a.B, a.L, a.H, a.dv), generator=gen).to(elem).to(dev)
            dS = torch.randn((a.B, a.H, a.dv, a.dk), generator=gen).to(dev)
            for _ in range(a.calls):
                gdn.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], dO, init_state=d["init_state"],
                              dfinal_state=dS)
    else:
        T = a.L if a.op == "decode_multi" else 1
        d = inputs.make_decode(a.B, a.H, a.dk, a.dv, T, a.dtype, seed=3)
        d = {k: v.to(dev) for k, v in d.items()}
        state = d["state0"].clone()
        # decode_multi takes [N, T, H, ...]; the generator gives [T, N, H, ...]
        m = {k: d[k].transpose(0, 1).contiguous() for k in ("q", "k", "v", "g", "beta")}
        for _ in range(a.calls):
            if a.op == "decode":
                gdn.decode_step(state, d["q"][0], d["k"][0], d["v"][0], d["g"][0], d["beta"][0])
            else:
                gdn.decode_multi(state, m["q"], m["k"], m["v"], m["g"], m["beta"])
    torch.cuda.synchronize()
    print(f"profile_case: {a.calls} x {a.op} done")


if __name__ == "__main__":
    main()
