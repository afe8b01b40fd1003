"""Run one product of the library a few times at one shape: the small, single-kernel
case that a profiler capture wants (``ncu -k regex:stream_kernel -s <skip> -c <n> ...``).

    python -m nvfp4_w4a16_moe_skinny_gb300.profile_case {lm_head,dense4096,dense14336,moe} M [REPS]

Weights are seeded N(0, 0.02) fp32 quantized on the GPU, activations N(0, 1)
bf16.  Each repetition launches one streaming kernel (lm_head, dense) or four
kernels (moe: route, gate+up, down, combine); the process exits non-zero if the
library's device error flag is set.
"""

from __future__ import annotations

import sys


def main(argv):
    import torch

    from nvfp4_w4a16_moe_skinny_gb300 import binding

    if len(argv) < 2:
        raise SystemExit(__doc__)
    kind, m = argv[0], int(argv[1])
    reps = int(argv[2]) if len(argv) > 2 else 3
    lib = binding.load()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)

    def randn(*shape):
        return torch.randn(shape, generator=g, device=dev)

    if kind == "moe":
        e, d, inter = 128, 2816, 704
        gu = lib.prepare(randn(e, 2 * inter, d) * 0.02, gated=True)
        dn = lib.prepare(randn(e, d, inter) * 0.02)
        sgu = lib.prepare(randn(2 * inter, d) * 0.02, gated=True)
        sdn = lib.prepare(randn(d, inter) * 0.02)
        x = randn(m, d).to(torch.bfloat16)
        logits = randn(m, e)
        torch.cuda.synchronize()
        for _ in range(reps):
            _, probs, offs, pairs = lib.route_topk(logits, 8)
            lib.moe_ffn(x, 8, probs, offs, pairs, gu, dn, sgu, sdn)
    else:
        shapes = {"lm_head": (262144, 2816), "dense4096": (4096, 4096), "dense14336": (14336, 4096)}
        if kind not in shapes:
            raise SystemExit(f"unknown case {kind!r}")
        n, k = shapes[kind]
        w = lib.prepare(randn(n, k) * 0.02)
        x = randn(m, k).to(torch.bfloat16)
        torch.cuda.synchronize()
        for _ in range(reps):
            if kind == "lm_head":
                lib.lm_head_argmax(w, x)
            else:
                lib.gemm(w, x)
    torch.cuda.synchronize()
    if lib.device_error() != 0:
        raise SystemExit("device error flag set")
    print(f"ok {kind} m={m} reps={reps}")


if __name__ == "__main__":
    main(sys.argv[1:])
