"""Profiling cases: eager calls of the library on seeded synthetic inputs, for
ncu captures of one kernel (the summaries under profiles/ name the command).

    python -m trellis_decode_gemv_gb300.profcase layer --shape 14336x4096 --K 2 --cb 0 --M 1
    python -m trellis_decode_gemv_gb300.profcase group --K 2 --cb 0 --M 1
    python -m trellis_decode_gemv_gb300.profcase group --K 2 --cb 1 --int8
    python -m trellis_decode_gemv_gb300.profcase group --K 2 --cb 0,1

`layer`: `--inst` distinct instances of one m x n layer (uniform random code
words, the input recipe's signs, scales and activations), `--calls` calls of
exl3_gemm_small in turn.  `group`: the Llama-3-8B layer set of one (K, code)
class (q, k, v, o, gate, up, down) as one exl3_gemm_grouped call (with
`--int8`, one exl3_gemm_int8act_grouped call; with several codes, the set once
per code in one exl3_gemm_multi call, or exl3_gemm_int8act_multi with
`--int8`), `--calls` times.  Nothing is checked here: the parity tests do that.
"""
import argparse

import torch

from . import binding as B
from . import synth

LLAMA8B_CLASS = [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096), (14336, 4096), (14336, 4096),
                 (4096, 14336)]


def _layer(m, n, K, M, seed, dev):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    words = (m // 16) * (n // 16) * 8 * K
    codes = torch.randint(-2**31, 2**31 - 1, (words,), generator=g, device=dev, dtype=torch.int64).to(torch.int32)
    return dict(codes=codes, m=m, n=n,
                s_in=torch.from_numpy(synth.sign_vector(n, seed + 1)).to(dev),
                s_out=torch.from_numpy(synth.sign_vector(m, seed + 2)).to(dev),
                scales=torch.from_numpy(synth.channel_scales(m, seed + 3)).to(dev),
                x=torch.from_numpy(synth.activations(M, n, seed + 4)).to(dev),
                y=torch.empty((M, m), dtype=torch.float16, device=dev))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("case", choices=["layer", "group"])
    ap.add_argument("--shape", default="14336x4096")
    ap.add_argument("--K", type=int, default=2)
    ap.add_argument("--cb", default="0", help="code, or a comma-separated list (group case: one multi-code call)")
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--inst", type=int, default=8)
    ap.add_argument("--calls", type=int, default=6)
    ap.add_argument("--path", choices=["auto", "shuffle", "tensor"], default="auto")
    ap.add_argument("--int8", action="store_true", help="group case on int8 activations (1MAD or mul1)")
    a = ap.parse_args(argv)
    cbs = [int(c) for c in a.cb.split(",")]
    a.cb = cbs[0]
    B.load_library()
    B.exl3_set_path({"auto": B.PATH_AUTO, "shuffle": B.PATH_SHUFFLE, "tensor": B.PATH_TENSOR}[a.path])
    dev = torch.device("cuda")
    if a.case == "layer":
        m, n = map(int, a.shape.split("x"))
        inst = [_layer(m, n, a.K, a.M, 1000 + 10 * i, dev) for i in range(a.inst)]
        ws = torch.zeros(B.exl3_workspace_bytes(m, n, a.M), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        for c in range(a.calls):
            L = inst[c % a.inst]
            B.exl3_gemm_small(L["codes"], a.K, a.cb, m, n, L["s_in"], L["s_out"], L["scales"], L["x"], y=L["y"],
                              workspace=ws)
        weights = m * n
    else:
        if len(cbs) > 1:
            layers = [dict(_layer(m, n, a.K, a.M, 3000 + 10 * i + 100 * c, dev), K=a.K, cb=c)
                      for c in cbs for i, (m, n) in enumerate(LLAMA8B_CLASS)]
            shapes = [(L["m"], L["n"]) for L in layers]
            if a.int8:
                ws = torch.zeros(B.exl3_multi_i8_workspace_bytes(shapes, a.M), dtype=torch.uint8, device=dev)
            else:
                ws = B.alloc_group_workspace(shapes, a.M, dev)

            def call(ls, K, cb, workspace):
                (B.exl3_gemm_int8act_multi if a.int8 else B.exl3_gemm_multi)(ls, workspace=workspace)
        else:
            layers = [_layer(m, n, a.K, a.M, 2000 + 10 * i, dev) for i, (m, n) in enumerate(LLAMA8B_CLASS)]
            if a.int8:
                ws = torch.zeros(B.exl3_group_i8_workspace_bytes(LLAMA8B_CLASS, a.M), dtype=torch.uint8, device=dev)
                call = B.exl3_gemm_int8act_grouped
            else:
                ws = B.alloc_group_workspace(LLAMA8B_CLASS, a.M, dev)
                call = B.exl3_gemm_grouped
        torch.cuda.synchronize()
        for _ in range(a.calls):
            call(layers, a.K, a.cb, workspace=ws)
        weights = sum(m * n for m, n in LLAMA8B_CLASS) * len(cbs)
    torch.cuda.synchronize()
    print(f"{a.case}: {a.calls} calls, {weights / 1e6:.1f} M weights each, K={a.K} code={','.join(map(str, cbs))} M={a.M}"
          f"{' int8' if a.int8 else ''}")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
