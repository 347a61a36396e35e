"""Benchmark: generated tokens/s at batch 1 on the Llama-3-8B-shaped workload.

One step = one greedy generation of 256 tokens (the first comes from the
prefill, which is outside the timed region; the other 255 come from
speculative cycles) with the static draft that skips 16 of 32 layers
(odd layers), draft length 6: K draft forwards, one verify pass over 7
rows, greedy acceptance and KV rollback per cycle.  Before every step the
request is rolled back to the end of its 512-token prompt, so each step
redoes the same generation from identical state.  Weights (16 GB bf16,
random, seeded) exceed L2 (129 MB) many times over, so no L2 flush is
needed between steps.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle
(the only reference this project has) on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "llama3_8b"
METRIC = "generated tokens/s at batch 1 (Llama-3-8B shape); verify-pass HBM GB/s"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1879.5)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def layer_bytes(cfg):
    hd, d, F = cfg.head_dim, cfg.d_model, cfg.ffn
    return 2 * (cfg.qkv_rows * d + d * cfg.n_q_heads * hd + 2 * F * d + d * F)


def pass_bytes(cfg, kept_layers, ctx, rows):
    """Algorithmic HBM bytes of one forward pass: weights of the layers run + lm_head,
    KV read for the visible context and KV written for the new rows.  The KV cache is
    fp32 (4 bytes per element), so its bytes count at 4 bytes; they are 0.7-1.6 % of a
    pass on these shapes."""
    kv_tok = 2 * cfg.n_kv_heads * cfg.head_dim * 4  # K and V, fp32, per layer per token
    return (kept_layers * layer_bytes(cfg) + 2 * cfg.vocab * cfg.d_model + kept_layers * kv_tok * (ctx + rows))


class Clocks:
    """nvidia-smi sampler for the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(ms: float, world: int, device: str = "cpu") -> float:
    """The slowest rank's time (the job's time when every rank runs its own replica)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


def run_ours(args):
    import numpy as np
    import torch

    import ssd_inputs as si
    import self_speculative_decoding_layer_gb300 as ssd

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()

    cfg = si.CONFIGS[WORKLOAD]
    weights = ssd.DeviceWeights(cfg)
    eng = ssd.Engine(cfg, weights)
    prompt = si.prompt(cfg)
    n_gen = cfg.n_gen
    eng.prefill(prompt)
    t0, p0 = eng.position()
    stream = eng.stream

    def step(kind=ssd.POLICY_STATIC):
        eng.rollback(t0, p0)
        return eng.generate(n_gen, kind)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize()

    def timed(fn, steps):
        barrier()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        outs = [fn() for _ in range(steps)]
        ev1.record(stream)
        barrier()
        ms = max_over_ranks(ev0.elapsed_time(ev1), world, "cuda")
        return ms, outs

    # warm-up (captures the graphs)
    for _ in range(args.warmup):
        ref_tokens = step()
    # speculative, timed, with per-pass CUDA-event timing
    eng.set_option(ssd.OPT_TIMING, 1)
    eng.reset_stats()
    clocks = Clocks(dev)
    clocks.start()
    ms, outs = timed(step, args.steps)
    clk = clocks.stop()
    st = eng.stats()
    pt = eng.pass_times()
    launches = st.get("launches", 0)
    eng.set_option(ssd.OPT_TIMING, 0)
    assert all(o == ref_tokens for o in outs), "generation is not deterministic"
    new_tokens = (n_gen - 1) * args.steps
    value = job_throughput(new_tokens, world, ms)

    # the library's own autoregressive path on the same request
    for _ in range(max(1, args.warmup // 2)):
        ar_tokens = step(ssd.POLICY_AR)
    ar_steps = max(1, args.steps // 2)
    ms_ar, ar_outs = timed(lambda: step(ssd.POLICY_AR), ar_steps)
    ar_value = (n_gen - 1) * ar_steps / (ms_ar / 1e3)
    lossless = ar_outs[0] == ref_tokens

    # end to end through the C ABI with host buffers: H2D prompt, prefill, generate, D2H tokens
    def e2e_step():
        eng.rollback(0, -1)
        eng.prefill(prompt)
        return eng.generate(n_gen, ssd.POLICY_STATIC)

    e2e_step()
    ms_e2e, _ = timed(e2e_step, max(1, args.steps // 2))
    e2e_value = job_throughput((n_gen - 1) * max(1, args.steps // 2), world, ms_e2e)

    # CLaSp DP pass at the end of that generation (target = the last accepted token; 16 of 32 layers
    # skipped, all j <= 16 batched per layer), CUDA events
    t_end, _ = eng.position()
    eng.dp_select(16)
    dp_steps = 3
    ms_dp, _ = timed(lambda: eng.dp_select(16), dp_steps)
    dp_bytes = cfg.n_layers * layer_bytes(cfg) + cfg.n_layers * 2 * cfg.n_kv_heads * cfg.head_dim * 4 * (t_end - 1)
    dp_gbs = dp_bytes / (ms_dp / dp_steps / 1e3) / 1e9

    # draft exit at the pages' best threshold (0.7): the same generation with each cycle's drafting cut
    # after the first draft whose top-1 probability is below 0.7, decided on the device.  The seeded
    # random weights give near-uniform next-token distributions (p1 far below 0.7), so every cycle
    # stops after one draft; the draft pass then runs 1 forward and 5 gated-off ones.  For scale: the
    # same loop with draft length 1.
    def exit_run(**kw):
        def one():
            eng.rollback(t0, p0)
            return eng.generate(n_gen, ssd.POLICY_STATIC, **kw)

        one()
        eng.set_option(ssd.OPT_TIMING, 1)
        eng.reset_stats()
        ms_x, outs_x = timed(one, max(1, args.steps // 2))
        stx, ptx = eng.stats(), eng.pass_times()
        eng.set_option(ssd.OPT_TIMING, 0)
        d_ms, d_n = ptx["draft"]
        return {"tokens_per_s": round((n_gen - 1) * max(1, args.steps // 2) / (ms_x / 1e3), 3),
                "lossless_vs_ar": outs_x[0] == ref_tokens,
                "mean_drafted": round(stx["drafted"] / max(stx["cycles"], 1), 4),
                "mean_accepted": round(stx["accepted"] / max(stx["cycles"], 1), 4),
                "draft_pass_ms": round(d_ms / max(d_n, 1), 4)}

    draft_exit = {"threshold": 0.7, **exit_run(exit_thr=0.7), "k1": exit_run(k=1)}

    # early exit ([CAS-blog] §2.2's fast level L1 on this shape): 70 % of the first 28 layers skipped
    # (nested around a 30 % set) and a 4-layer early exit, so 8 of 32 layers run per draft forward
    l1_skip = si.cascade_levels(cfg.n_layers, 4)[0][0]
    early = exit_run(skip=l1_skip, early_exit=4)
    l1_kept = cfg.n_layers - len(set(l1_skip) | set(range(cfg.n_layers - 4, cfg.n_layers)))
    l1_bytes = sum(pass_bytes(cfg, l1_kept, cfg.prompt_len + n_gen // 2 + r, 1) for r in range(cfg.draft_k))
    early["layers_run"] = l1_kept
    early["draft_pass_gbs"] = round(l1_bytes / (early["draft_pass_ms"] / 1e3) / 1e9, 1)

    # DyTC against the horizontal and vertical cascade baselines ([CAS-paper] abstract: DyTC +47 % over cascade
    # baselines on trained models) with the cascade levels of this shape (L1 70 % skipped, L2 30 % + int8,
    # L3 int8): the same greedy output, tokens/s of each (the random weights accept no draft, so this
    # compares the cost of each scheme's drafting when drafts fail)
    levels = si.cascade_levels(cfg.n_layers)

    def cascade_run(kind, **kw):
        def one():
            eng.rollback(t0, p0)
            return eng.generate(n_gen, kind, levels=levels, **kw)

        one()
        eng.reset_stats()
        ms_c, outs_c = timed(one, 1)
        stc = eng.stats()
        return {"tokens_per_s": round((n_gen - 1) / (ms_c / 1e3), 3), "lossless_vs_ar": outs_c[0] == ref_tokens,
                "cycles": stc["cycles"], "mean_drafted": round(stc["drafted"] / max(stc["cycles"], 1), 3)}

    cascades = {"levels": "L1 skip 70 %, L2 skip 30 % + int8, L3 int8", "dytc": cascade_run(ssd.POLICY_DYTC),
                "hcascade_2_2_2": cascade_run(ssd.POLICY_HCASCADE, hc_len=(2, 2, 2)),
                "vcascade_L1_to_L2_k6": cascade_run(ssd.POLICY_VCASCADE, k=6, vc_lo=0, vc_hi=1)}

    # latency model ([CAS-blog] §3.2: latency = b0 + b1 seq_len + b2 layer_depth), fitted from CUDA-event
    # timings of one-draft passes on three context lengths and checked on the three between them
    # (the pages report < 15 % error on an A100).  Rolls the context back, so it runs last.
    def latency_model(int8):
        eng.rollback(0, -1)
        eng.prefill(prompt)
        eng.decode_ar(n_gen)  # a context of prompt + n_gen tokens for the grid
        t_now, _ = eng.position()
        seqs = [s_ for s_ in (768, 640, 512, 384, 256, 128) if s_ <= t_now]
        depths = [4, 8, 16, 24, 32]
        train = np.zeros((len(seqs), len(depths)), dtype=np.uint8)
        train[0::2] = 1
        beta, times = eng.calibrate_latency(depths, seqs, act_int8=int8, reps=5, train=train)
        S = np.repeat(seqs, len(depths)).reshape(len(seqs), len(depths))
        D = np.tile(depths, (len(seqs), 1))
        err = np.abs(beta[0] + beta[1] * S + beta[2] * D - times) / times
        held = err[train == 0]
        return {"beta_ms": [float(b) for b in beta], "seq_lens": seqs, "depths": depths,
                "train": "seq_lens 768, 512, 256 (all depths)",
                "heldout_mean_rel_err": round(float(held.mean()), 4),
                "heldout_max_rel_err": round(float(held.max()), 4)}

    # device timeline (%globaltimer per kernel) of one draft pass: per-kernel duration and GB/s
    eng.rollback(t0, p0)
    eng.set_option(ssd.OPT_TRACE, 1)
    eng.draft(cfg.skip, cfg.draft_k)
    trace = eng.trace()
    eng.set_option(ssd.OPT_TRACE, 0)
    eng.rollback(t0, p0)
    timeline = kernel_timeline(cfg, trace)
    lat_model = {"bf16": latency_model(False), "int8": latency_model(True), "pages_bound": 0.15}

    # roofline: draft and verify passes (algorithmic bytes / CUDA-event pass time)
    hbm, _, peak_kind = peaks()
    kept = cfg.n_layers - len(cfg.skip)
    ctx_mid = cfg.prompt_len + n_gen // 2
    draft_ms, n_draft = pt["draft"]
    verify_ms, n_verify = pt["verify"]
    k = cfg.draft_k
    draft_bytes = sum(pass_bytes(cfg, kept, ctx_mid + r, 1) for r in range(k))  # one draft pass = K forwards
    # DRAM bytes ncu measured (dram__bytes_read.sum + dram__bytes_write.sum over every launch of one draft
    # forward of the 8B shape cut to 4 layers, at this workload's 512-token context: 1944.13 MB) over that
    # forward's algorithmic bytes (1931.49 MB): the pass moves what the method needs plus 0.65 %.  Scaled to
    # this pass by its algorithmic bytes.
    traffic_ratio = 1.0065
    verify_bytes = pass_bytes(cfg, cfg.n_layers, ctx_mid, k + 1)
    ar_gbs = pass_bytes(cfg, cfg.n_layers, ctx_mid, 1) * ar_value / 1e9  # one full forward per AR token
    draft_gbs = draft_bytes / (draft_ms / max(n_draft, 1) / 1e3) / 1e9 if n_draft else None
    verify_gbs = verify_bytes / (verify_ms / max(n_verify, 1) / 1e3) / 1e9 if n_verify else None
    cycles = st["cycles"]
    mean_acc = st["accepted"] / cycles if cycles else 0.0

    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded random weights N(0,0.02), uniform random prompt ids)",
        "config": {"workload": "Llama-3-8B shape (32 layers, d 4096, 32q/8kv heads, ffn 14336, vocab 128256), "
                               "prompt 512, generate 256, static skip 16/32 (odd layers), draft length 6, batch 1",
                   "l2": "inputs larger than L2 (16 GB of weights streamed per pass); no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "precision": "bf16 weights; fp32 KV cache, activations and accumulation "
                                "(algorithmic bytes count the KV cache at 4 bytes per element)"},
        "verify_pass_gbs": round(verify_gbs, 1) if verify_gbs else None,
        "draft_pass_gbs": round(draft_gbs, 1) if draft_gbs else None,
        "ar_tokens_per_s": round(ar_value, 3),
        "ar_pass_gbs": round(ar_gbs, 1),
        "ar_pass_frac": round(ar_gbs / hbm, 4),
        "speedup_vs_ar": round(value / ar_value, 4),
        "lossless_vs_ar": lossless,
        "mean_accepted": round(mean_acc, 4),
        "cycles_per_step": cycles / args.steps,
        "draft_exit": draft_exit,
        "early_exit": early,
        "latency_model": lat_model,
        "cascades": cascades,
        "e2e": {"value": round(e2e_value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 4 * cfg.prompt_len,
                "d2h_bytes_per_step": 4 * n_gen},
        "gpu_launches": launches,
        "roofline": {"bound": "hbm",
                     "kernel": "draft pass: one CUDA graph of K=6 batch-1 forwards over the 16 kept layers "
                               "(k_gemv_rs weight streaming, k_attention, lm_head + k_argmax), CUDA events on the "
                               "engine stream over the timed region",
                     "achieved": round(draft_gbs, 1) if draft_gbs else None, "peak": hbm, "unit": "GB/s",
                     "frac": round(draft_gbs / hbm, 4) if draft_gbs else None, "peak_kind": peak_kind,
                     "algorithmic_bytes": int(draft_bytes),
                     "traffic": int(draft_bytes * traffic_ratio),
                     "verify": {"kernel": "verify pass: 7 rows through all 32 layers (k_mma tcgen05, k_attention)",
                                "achieved": round(verify_gbs, 1) if verify_gbs else None,
                                "frac": round(verify_gbs / hbm, 4) if verify_gbs else None,
                                "algorithmic_bytes": int(verify_bytes)},
                     "dp": {"kernel": "CLaSp DP pass: 17 rows per layer, 32 layers (k_mma, k_attention, k_dp_step)",
                            "achieved": round(dp_gbs, 1), "frac": round(dp_gbs / hbm, 4),
                            "algorithmic_bytes": int(dp_bytes), "ms": round(ms_dp / dp_steps, 3)},
                     "timeline": timeline},
        "clocks": clk,
    }
    if not args.main_only:
        # the other workloads, one after the other on the same GPU (the 8B weights are shared with the
        # CLaSp workload and freed before the 13B and 70B models are built)
        extra = {"llama3_8b_clasp": workload_entry("llama3_8b_clasp", hbm, weights)}
        del eng, weights
        import gc

        gc.collect()
        torch.cuda.empty_cache()
        for name in ("llama2_13b_cascade", "llama3_70b_clasp"):
            extra[name] = workload_entry(name, hbm)
            gc.collect()
            torch.cuda.empty_cache()
        line["workloads"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def workload_entry(name, hbm, weights=None):
    """One untimed and one timed generation of a workload with its own policy, then its autoregressive
    baseline: tokens/s, speedup over the library's own AR path, mean accepted drafts, and per-pass GB/s with
    the fraction of the measured HBM peak (CUDA events around each pass, engine stream)."""
    import torch

    import ssd_inputs as si
    import self_speculative_decoding_layer_gb300 as ssd

    cfg = si.CONFIGS[name]
    t_load = time.time()
    w = weights if weights is not None else ssd.DeviceWeights(cfg)
    eng = ssd.Engine(cfg, w)
    prompt = si.prompt(cfg)
    eng.prefill(prompt)
    load_s = time.time() - t_load
    t0, p0 = eng.position()
    n_gen = cfg.n_gen
    if cfg.tree:
        kind, kw = ssd.POLICY_DYTC, {"levels": cfg.levels}
        desc = "DyTC tree (<= 16 nodes, depth <= 6) over the three cascade levels, EMA alpha 0.2"
    else:
        kind, kw = ssd.POLICY_CLASP, {"k": cfg.draft_k, "dp_n_skip": cfg.dp_n_skip, "dp_interval": cfg.dp_interval}
        desc = (f"CLaSp: DP for {cfg.dp_n_skip} of {cfg.n_layers} layers after prefill and every "
                f"{cfg.dp_interval} verify steps, draft length {cfg.draft_k}")

    def gen(kd, n, **k2):
        # back to the end of the prompt; the last prompt token is run again so that it is the CLaSp target
        eng.rollback(t0 - 1)
        eng.prefill([int(prompt[-1])])
        if cfg.tree:  # every generation starts from the initial acceptance estimates
            eng.set_ema([cfg.ema_init] * len(cfg.levels))
        return eng.generate(n, kd, **k2)

    def timed(fn):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(eng.stream)
        out = fn()
        b.record(eng.stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b), out

    gen(kind, min(n_gen, 3 * (cfg.draft_k + 1)), **kw)  # captures the passes' graphs
    eng.set_option(ssd.OPT_TIMING, 1)
    eng.reset_stats()
    ms, toks = timed(lambda: gen(kind, n_gen, **kw))
    st, pt = eng.stats(), eng.pass_times()
    eng.set_option(ssd.OPT_TIMING, 0)
    n_ar = min(n_gen, 96)
    gen(ssd.POLICY_AR, 8)
    ms_ar, ar_toks = timed(lambda: gen(ssd.POLICY_AR, n_ar))
    value = (n_gen - 1) / (ms / 1e3)
    ar_value = (n_ar - 1) / (ms_ar / 1e3)
    cycles = max(st["cycles"], 1)
    ctx_mid = cfg.prompt_len + n_gen // 2
    out = {"workload": f"{name}: {cfg.n_layers} layers, d {cfg.d_model}, {cfg.n_q_heads}q/{cfg.n_kv_heads}kv heads, "
                       f"ffn {cfg.ffn}, vocab {cfg.vocab}, {cfg.dtype}; prompt {cfg.prompt_len}, generate {n_gen}; "
                       + desc,
           "tokens_per_s": round(value, 3), "ar_tokens_per_s": round(ar_value, 3),
           "speedup_vs_ar": round(value / ar_value, 4), "lossless_vs_ar": toks[:n_ar] == ar_toks,
           "mean_accepted": round(st["accepted"] / cycles, 4), "cycles": st["cycles"],
           "dp_runs": st["dp_runs"], "setup_s": round(load_s, 1)}
    full = pass_bytes(cfg, cfg.n_layers, ctx_mid, 1)
    out["ar_pass_gbs"] = round(full * ar_value / 1e9, 1)
    out["ar_pass_frac"] = round(full * ar_value / 1e9 / hbm, 4)
    d_ms, d_n = pt["draft"]
    v_ms, v_n = pt["verify"]
    dp_ms, dp_n = pt["dp"]
    if kind == ssd.POLICY_CLASP:
        kept = cfg.n_layers - cfg.dp_n_skip
        db = sum(pass_bytes(cfg, kept, ctx_mid + r, 1) for r in range(cfg.draft_k))
        vb = pass_bytes(cfg, cfg.n_layers, ctx_mid, cfg.draft_k + 1)
        if d_n:
            g = db / (d_ms / d_n / 1e3) / 1e9
            out["draft_pass"] = {"ms": round(d_ms / d_n, 3), "gbs": round(g, 1), "frac": round(g / hbm, 4)}
        if dp_n:
            kv = cfg.n_layers * 2 * cfg.n_kv_heads * cfg.head_dim * 4 * ctx_mid
            g = (cfg.n_layers * layer_bytes(cfg) + kv) / (dp_ms / dp_n / 1e3) / 1e9
            out["dp_pass"] = {"ms": round(dp_ms / dp_n, 3), "rows": cfg.dp_n_skip + 1, "gbs": round(g, 1),
                              "frac": round(g / hbm, 4)}
    else:
        rows = round(st["drafted"] / cycles) + 1
        vb = pass_bytes(cfg, cfg.n_layers, ctx_mid, rows)
        out["draft_expansions_per_cycle"] = round(d_n / cycles, 3)
        out["draft_ms_per_cycle"] = round(d_ms / cycles, 3)
        out["mean_tree_rows"] = rows
    if v_n:
        g = vb / (v_ms / v_n / 1e3) / 1e9
        out["verify_pass"] = {"ms": round(v_ms / v_n, 3), "gbs": round(g, 1), "frac": round(g / hbm, 4)}
    eng.close()
    del eng
    return out


def kernel_timeline(cfg, trace):
    """Median device time (from the first CTA past its dependency wait to the last CTA's end, %globaltimer)
    of each projection of a traced draft pass, with its weight bytes per microsecond."""
    hd, d, F = cfg.head_dim, cfg.d_model, cfg.ffn
    wbytes = {"qkv": 2 * cfg.qkv_rows * d, "o": 2 * d * cfg.n_q_heads * hd, "gate_up": 4 * F * d, "down": 2 * d * F,
              "lm_head": 2 * cfg.vocab * d}
    kinds = {2: "attention", 10: "qkv", 12: "gate_up", 13: "lm_head"}
    per = {}
    prev = None
    for kind, _res, run, end in trace:
        if run <= 0 or end <= run:
            continue
        name = kinds.get(kind)
        if kind == 11:
            name = "o" if prev == "attention" else "down"
        if name is None:
            continue
        per.setdefault(name, []).append((end - run) / 1e3)
        prev = name
    out = {}
    for name, v in per.items():
        us = statistics.median(v)
        e = {"launches": len(v), "median_us": round(us, 2)}
        if name in wbytes:
            e["gbs"] = round(wbytes[name] / us / 1e3, 1)
        out[name] = e
    return {"unit": "us / GB/s", "source": "device timeline (%globaltimer) of one traced draft pass", **out}


def oracle_sample(layers_sample=4, decode_steps=2):
    """Time the CPU oracle on a bounded sample of the workload: the 8B-shaped model cut
    to `layers_sample` layers, prefill of the 512-token prompt (untimed), then
    `decode_steps` greedy decode steps (timed).  The per-token time is scaled to the
    full depth: t_token = t_lm_head + 32/layers_sample * (t_step - t_lm_head)."""
    import numpy as np

    import ssd_inputs as si
    from oracle import decode, model

    cfg = si.CONFIGS[WORKLOAD]
    cut = cfg.replace(n_layers=layers_sample)
    W = model.Weights(cut)
    sess = decode.Session(W, cfg.max_ctx)
    sess.prefill(si.prompt(cfg))
    for i in range(layers_sample):
        W.layer(i)
    t_steps = []
    for _ in range(decode_steps):
        t0 = time.perf_counter()
        sess.ar_step()
        t_steps.append(time.perf_counter() - t0)
    x = np.zeros((1, cfg.d_model))
    t0 = time.perf_counter()
    W.logits(x)
    t_lm = time.perf_counter() - t0
    t_step = min(t_steps)
    t_token = t_lm + cfg.n_layers / layers_sample * max(t_step - t_lm, 0.0)
    return 1.0 / t_token, t_token


def cpu_baseline(args):
    cores = os.cpu_count()
    v, t_token = oracle_sample()
    return {"value": round(v, 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "numpy float64 oracle, greedy decode at context 512 of the 8B shape cut to 4 layers "
                      f"(2 timed steps after an untimed 512-token prefill), per-token time scaled to 32 layers "
                      f"+ lm_head: {t_token:.2f} s/token; BLAS threads = all {cores} cores"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = os.cpu_count()
    t0 = time.time()
    vals = []
    for _ in range(max(1, args.steps)):
        v, t_token = oracle_sample(decode_steps=1)
        vals.append(v)
    value = statistics.median(vals)
    wall = time.time() - t0
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 / value, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded random weights, uniform random prompt ids)",
            "config": {"workload": "Llama-3-8B shape, prompt 512, greedy decode (autoregressive on the oracle)"},
            "cpu_baseline": {"value": round(value, 5), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "per step: 8B shape cut to 4 layers, 512-token prefill untimed, one decode "
                                       "step timed, scaled to 32 layers + lm_head"},
            "e2e": {"value": round(value, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 1)}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--main-only", action="store_true", help="skip the 13B, 8B-CLaSp and 70B workload entries")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
