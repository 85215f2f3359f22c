"""Small, self-contained launches of one library kernel each, for profilers
(ncu captures one launch of a case run a few times).

  python -m ulysses_sequence_attention_tf_gb300.profile_cases projection [--S 8192] [--iters 3]
  python -m ulysses_sequence_attention_tf_gb300.profile_cases scatter_fused [--S 32760] [--iters 3]
  python -m ulysses_sequence_attention_tf_gb300.profile_cases scatter_fused_qk [--S 32760] [--iters 3]
  python -m ulysses_sequence_attention_tf_gb300.profile_cases scatter --S 4096 --H 24 --layout fused
  python -m ulysses_sequence_attention_tf_gb300.profile_cases gather --P 8 --H 48 --D 64 --B 2 --S 6008
  python -m ulysses_sequence_attention_tf_gb300.profile_cases rope_table [--S 32760] [--iters 3]

``--layout``: v_strided (Q/K contiguous, V a view into a fused projection; the
default), fused (Q/K/V all views of one fused projection), contiguous, pad16
(every head row followed by 16 bytes of padding: sources only 16-byte aligned,
which sends fused scatters to the register kernel).  ``rope_table`` builds the
resident cos/sin table of (theta, S, D) once per iteration, each time for
another theta.

Inputs are the seeded synthetic ones of ``synth``; shapes default to the
video-DiT workload's head geometry (P=4, H=40, D=128, bf16) with a smaller
sequence for the projection, so a capture holds well under a few GB.
"""
from __future__ import annotations

import argparse

import torch

from . import binding, build, synth


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("case", choices=["projection", "scatter", "scatter_fused", "scatter_fused_qk", "gather",
                                     "rope_table"])
    ap.add_argument("--P", type=int, default=4)
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--S", type=int, default=None, help="global tokens (default 8192 projection, 32760 others)")
    ap.add_argument("--H", type=int, default=40)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--rope", choices=["interleaved", "neox"], default="interleaved")
    ap.add_argument("--layout", choices=["v_strided", "fused", "contiguous", "pad16"], default="v_strided")
    ap.add_argument("--dtype", choices=["bf16", "fp16"], default="bf16", help="element type of the scatters")
    args = ap.parse_args(argv)
    P, H, D, B = args.P, args.H, args.D, args.B
    S = args.S or (8192 if args.case == "projection" else 32760)
    Sl, Hl = S // P, H // P
    build.build()
    binding.lib()
    binding.use_torch_allocator(True)
    dev = torch.device("cuda", 0)
    dt = torch.float16 if args.dtype == "fp16" and args.case != "projection" else torch.bfloat16
    wq, wk = synth.norm_weights(D, dt, seed=0, device=dev)
    if args.case == "projection":
        xs, w = synth.projection_inputs(P, B, Sl, H * D, H, D, torch.bfloat16, seed=1, device=dev)
        outs = {k: [torch.empty((B, S, Hl, D), dtype=torch.bfloat16, device=dev) for _ in range(P)] for k in "qkv"}

        def call():
            binding.project_qkv_into(xs, w, H, outs["q"], outs["k"], outs["v"], norm_rope=True, q_weight=wq,
                                     k_weight=wk, rope=args.rope)
    elif args.case == "rope_table":
        it = iter(range(args.iters))

        def call():
            binding.rope_table(10000.0 + next(it), S, D)
    elif args.case in ("scatter", "scatter_fused", "scatter_fused_qk"):
        if args.layout == "pad16":
            pad = 16 // 2
            g = {key: [synth.qkv_shards(1, B, Sl, H, D + pad, dt, seed=10 * r + i, device=dev,
                                        with_k=False, with_v=False)["q"][0][..., :D] for r in range(P)]
                 for i, key in enumerate("qkv")}
        else:
            g = synth.qkv_shards(P, B, Sl, H, D, dt, seed=0, layout=args.layout, device=dev)
        v = None if args.case == "scatter_fused_qk" else g["v"]  # Q/K only: V moves elsewhere
        fused = args.case != "scatter"

        def call():
            if fused:
                binding.scatter_qkv("profile", g["q"], g["k"], v, norm_rope=True, q_weight=wq, k_weight=wk,
                                    rope=args.rope)
            else:
                binding.scatter_qkv("profile", g["q"], g["k"], v)
    else:
        attn = synth.attn_outputs(P, B, S, Hl, D, torch.bfloat16, seed=0, device=dev)

        def call():
            binding.gather_out("profile", attn)
    for _ in range(args.iters):
        call()
    torch.cuda.synchronize()
    print(f"{args.case}: {args.iters} launches, device status {binding.device_status()}")


if __name__ == "__main__":
    main()
