"""Run a few decode passes of a workload for profiling (e.g. under ncu).

    python -m self_speculative_decoding_layer_gb300.profile_passes --workload llama3_8b --cycles 1

Prefills the workload's prompt (or --prompt tokens of it), runs one
untimed cycle that captures the CUDA graphs, then `--cycles` speculative
cycles (draft pass of draft_k layer-skipped forwards, verify pass,
acceptance) with the workload's static skip set, `--ar` autoregressive
steps and `--dp-runs` CLaSp DP searches for `--dp` skipped layers (one
untimed first), each group inside an NVTX range for ncu's --nvtx filters.
"""
import argparse
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def main():
    import torch

    import ssd_inputs as si
    import self_speculative_decoding_layer_gb300 as ssd

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama3_8b")
    ap.add_argument("--cycles", type=int, default=1)
    ap.add_argument("--ar", type=int, default=1)
    ap.add_argument("--prompt", type=int, default=0, help="prompt length (0 = the workload's)")
    ap.add_argument("--gemm-impl", type=int, default=0)
    ap.add_argument("--pdl", type=int, default=1)
    ap.add_argument("--layers", type=int, default=0, help="cut the model to this many layers (0 = all)")
    ap.add_argument("--dp", type=int, default=0, help="CLaSp DP searches for this many skipped layers (0 = none)")
    ap.add_argument("--dp-runs", type=int, default=1)
    args = ap.parse_args()
    cfg = si.CONFIGS[args.workload]
    if args.layers:
        cfg = cfg.replace(n_layers=args.layers, skip=tuple(i for i in cfg.skip if i < args.layers))
    # a cross-check kernel (--gemm-impl 1..5) runs on the test library
    eng = ssd.Engine(cfg, ssd.DeviceWeights(cfg), xcheck=args.gemm_impl != 0)
    eng.set_option(ssd.OPT_GEMM_IMPL, args.gemm_impl)
    eng.set_option(ssd.OPT_PDL, args.pdl)
    nvtx = torch.cuda.nvtx  # ranges "prefill", "cycles", "ar", "dp" (ncu --nvtx --nvtx-include "<name>/")
    torch.cuda.synchronize()
    nvtx.range_push("prefill")
    eng.prefill(si.prompt(cfg, args.prompt or cfg.prompt_len))
    torch.cuda.synchronize()
    nvtx.range_pop()
    skip = cfg.skip if (cfg.skip or args.layers) else tuple(range(1, cfg.n_layers, 2))
    t, p = eng.position()
    eng.verify([p] + eng.draft(skip, cfg.draft_k))  # captures the passes' graphs
    torch.cuda.synchronize()
    nvtx.range_push("cycles")
    for _ in range(args.cycles):
        t, p = eng.position()
        eng.verify([p] + eng.draft(skip, cfg.draft_k))
    torch.cuda.synchronize()
    nvtx.range_pop()
    if args.ar:
        eng.decode_ar(1)
        torch.cuda.synchronize()
        nvtx.range_push("ar")
        eng.decode_ar(args.ar)
        torch.cuda.synchronize()
        nvtx.range_pop()
    if args.dp:
        eng.dp_select(args.dp)
        torch.cuda.synchronize()
        nvtx.range_push("dp")
        for _ in range(args.dp_runs):
            eng.dp_select(args.dp)
        torch.cuda.synchronize()
        nvtx.range_pop()
    torch.cuda.synchronize()
    print("done", eng.position(), eng.stats()["launches"])


if __name__ == "__main__":
    main()
