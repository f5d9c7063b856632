#!/usr/bin/env python
"""Throughput of the diagonal-batched ARMT forward pass on GB300.

One step = one forward pass over the whole workload (default: ARMT-1B shape,
128 segments x 1024 tokens = 131,072 tokens, batch 1, diagonal schedule),
inputs already resident in HBM.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-seq] [--no-cpu] [--no-e2e]
                  [--no-full] [--no-microbatch] [--no-split] [--no-wavefront]
                  [--no-backward]

Inside the timed region only the roofline kernel (the gate-up GEMM) carries
per-launch CUDA events; the per-kernel-class table comes from one more forward
after it.  Besides the timed forward the line reports the sequential schedule,
the uniform-load bound, the LM head, the full-attention LLaMA on the same
weights, diagonal batching vs micro-batching, the split-precision mode
(activations as bf16 high + low parts), the persistent wavefront schedule
against per-diagonal launches on an fp32 model, the backward pass on the same
fp32 model, the end-to-end host-buffer path, device memory, and the oracle on
the host cores.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (one segment through every layer per step).
Under torchrun each rank runs an independent replica (weak scaling); the
path has no exchange step, so there is no collective in the data path.
"""
import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/sec ARMT-1B @131072 tok (1 GB300)"
UNIT = "tokens/s"


def metric_name(workload):
    return METRIC if workload == "armt-1b-131k" else f"tokens/sec {workload} (1 GB300)"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default="armt-1b-131k")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-seq", action="store_true", help="skip the sequential-schedule comparison")
    p.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-full", action="store_true",
                   help="skip the full-causal-attention LLaMA baseline on the same weights")
    p.add_argument("--no-microbatch", action="store_true",
                   help="skip the diagonal-batching vs micro-batching comparison")
    p.add_argument("--no-split", action="store_true",
                   help="skip the split-precision (bf16 high + low activations) forward")
    p.add_argument("--no-backward", action="store_true",
                   help="skip the backward-pass timing (fp32 model)")
    p.add_argument("--no-wavefront", action="store_true",
                   help="skip the persistent-wavefront comparison (fp32 model)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def cell_flops(cfg):
    """Algorithmic FLOPs of one cell, split by kernel class (multiply-add = 2)."""
    T, d, F = cfg.rows, cfg.d_model, cfg.ffn_dim
    Hq, Hkv, hd, k, P, M = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.key_dim, cfg.phi_dim, cfg.n_mem
    return {
        "gemm_qkv": 2.0 * T * d * (Hq + 2 * Hkv) * hd,
        "gemm_o": 2.0 * T * Hq * hd * d,
        "gemm_gateup": 2.0 * T * d * 2 * F,
        "gemm_down": 2.0 * T * F * d,
        "attention": 4.0 * Hq * hd * T * (T + 1) / 2.0,
        "assoc_read": 2.0 * T * d * k + 2.0 * T * P * d,
        "assoc_write": 2.0 * M * d * (k + 1 + d) + 4.0 * M * P * d,
    }


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        return self

    def __exit__(self, *a):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()

    def summary(self):
        self.f.flush()
        rows = []
        try:
            with open(self.f.name) as fh:
                for line in fh:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
        finally:
            os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


def replica_throughput(ms_local, n_tok_local, steps, world, dist=None, device="cpu"):
    """Whole-job throughput of `world` independent replicas (weak scaling).

    Each rank ran `steps` steps over `n_tok_local` tokens in `ms_local` ms;
    the job's time is the slowest rank's (all-reduce MAX), its work the sum
    over ranks.  Returns (max_ms, tokens_per_s).
    """
    ms = float(ms_local)
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * n_tok_local * steps / (ms / 1000.0)


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def oracle_sample_seconds(cfg, W, tokens, n_seg=1):
    """fp64 oracle on the first n_seg segments through every layer; returns seconds."""
    from oracle import armt_oracle as O
    t0 = time.perf_counter()
    O.forward(cfg, W, tokens[:n_seg * cfg.seg_len], n_seg)
    return time.perf_counter() - t0


def run_reference(args, rank):
    """--impl reference: the oracle as it stands, on the host cores."""
    from recurrent_memory_transformer_gb300 import inputs as I
    if rank != 0:
        return
    cfg, n_seg, seed = I.WORKLOADS[args.workload]
    # 3B/8B: one layer of the same shape, timed and scaled by the layer count
    # (every layer costs the same), so that a step stays within seconds
    big = args.workload in I.DEVICE_WEIGHT_WORKLOADS
    cfg_s = dataclasses.replace(cfg, n_layers=1) if big else cfg
    scale = cfg.n_layers if big else 1
    W = I.make_weights(cfg_s, seed)
    tok = I.make_tokens(cfg, n_seg, seed)
    for _ in range(args.warmup):
        oracle_sample_seconds(cfg_s, W, tok)
    ts = [oracle_sample_seconds(cfg_s, W, tok) * scale for _ in range(args.steps)]
    tok_per_step = cfg.seg_len
    value = tok_per_step * len(ts) / sum(ts)
    cores = os.cpu_count()
    sample = (f"fp64 oracle, segment 0 ({cfg.seg_len} tokens) through all {cfg.n_layers} layers per step; "
              "per-segment cost is constant in the segment recurrence")
    if big:
        sample = (f"fp64 oracle, segment 0 ({cfg.seg_len} tokens) through one layer of this shape, "
                  f"x {cfg.n_layers} layers per step; per-segment cost is constant in the recurrence")
    print(json.dumps({
        "impl": "reference", "metric": metric_name(args.workload), "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * sum(ts) / len(ts),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "tokens": n_seg * cfg.seg_len},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank)

    import numpy as np
    import torch

    from recurrent_memory_transformer_gb300 import armt as B
    from recurrent_memory_transformer_gb300 import build as build_mod
    from recurrent_memory_transformer_gb300 import inputs as I

    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    if rank == 0:
        build_mod.build()
    if pg is not None:
        pg.barrier()
    B.load_library()

    cfg, n_seg, seed = I.WORKLOADS[args.workload]
    tok_np = I.make_tokens(cfg, n_seg, seed)
    if args.workload in I.DEVICE_WEIGHT_WORKLOADS:
        W = None   # drawn on the GPU; the oracle baseline needs host weights
        model = B.Model(cfg, I.make_weights_device(cfg, seed))
    else:
        W = I.make_weights(cfg, seed)
        model = B.Model(cfg, B.device_weight_tensors(cfg, W))
    torch.cuda.empty_cache()   # the caller's weight copies are no longer needed
    tokens = torch.from_numpy(tok_np).cuda()
    n_tok = n_seg * cfg.seg_len
    hidden = torch.empty((n_tok, cfg.d_model), dtype=torch.float32, device="cuda")
    A = torch.empty(model.a_elems, dtype=torch.float32, device="cuda")
    z = torch.empty(model.z_elems, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    ws_create = model.armt_memory_bytes()[1]

    def step(schedule=B.SCHEDULE_DIAGONAL):
        model.armt_forward(tokens, n_seg, hidden, A, z, 0, stream, schedule)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    model.armt_sync_status()

    # ---- timed region: K steps, CUDA events on the launch stream ----------
    # only the roofline kernel (gate-up GEMM) gets per-launch events here, so
    # that the events disturb the timed forward as little as possible; the
    # per-class breakdown comes from one more forward after the timed region
    model.armt_set_profiling_mask(["gemm_gateup"])
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    if pg is not None:
        pg.barrier()
    ms_total = ev0.elapsed_time(ev1)
    kt_timed = model.armt_kernel_times()
    model.armt_set_profiling(True)
    step()
    kt = model.armt_kernel_times()          # one forward, every class
    model.armt_set_profiling(False)
    model.armt_sync_status()
    ms_total, value = replica_throughput(ms_total, n_tok, args.steps, world, pg, "cuda")
    clocks = clk.summary()
    ms_step = ms_total / args.steps

    # ---- roofline of the dominant kernel (gate-up grouped GEMM) ----------
    peaks, peak_src = load_peaks()
    fl = cell_flops(cfg)
    cells = cfg.n_layers * n_seg * args.steps
    gu_launches, gu_ms = kt_timed["gemm_gateup"]
    gu_tflops = fl["gemm_gateup"] * cells / (gu_ms / 1000.0) / 1e12 if gu_ms > 0 else None
    peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
    # DRAM bytes of the gate-up GEMM per cell: dram__bytes_read.sum +
    # dram__bytes_write.sum of one ncu capture of an 8-cell launch of the
    # current kernel (ARMT-1B, 8 segments), divided by 8.  Traffic scales with
    # cells (each cell's layer weights + activations), so per launch it is
    # this times the launch's cells.  None until a capture of the current
    # kernel exists.
    GATEUP_DRAM_BYTES_PER_CELL_1B = 86.5e6
    gu_traffic = (GATEUP_DRAM_BYTES_PER_CELL_1B * cells / gu_launches
                  if (GATEUP_DRAM_BYTES_PER_CELL_1B and gu_launches and args.workload.startswith("armt-1b"))
                  else None)
    cells1 = cfg.n_layers * n_seg           # cells of the one profiled forward
    gemm_keys = ("gemm_qkv", "gemm_o", "gemm_gateup", "gemm_down")
    gemm_ms = sum(kt[k][1] for k in gemm_keys)
    gemm_tflops = sum(fl[k] for k in gemm_keys) * cells1 / (gemm_ms / 1000.0) / 1e12 if gemm_ms else None
    total_flops = sum(fl.values()) * cfg.n_layers * n_seg
    per_class = {k: {"launches": int(v[0]), "ms_per_step": v[1],
                     "tflops": (fl[k] * cells1 / (v[1] / 1000.0) / 1e12) if (k in fl and v[1] > 0) else None}
                 for k, v in kt.items()}

    # ---- sequential schedule on the same inputs (speed-up denominator) ---
    seq = None
    if not args.no_seq:
        step(B.SCHEDULE_SEQUENTIAL)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step(B.SCHEDULE_SEQUENTIAL)
        e1.record(stream)
        torch.cuda.synchronize()
        seq_ms = e0.elapsed_time(e1)
        seq = {"ms_per_step": seq_ms, "tokens_per_s": n_tok / (seq_ms / 1000.0),
               "speedup_diag_over_seq": seq_ms / ms_step}

    # ---- ideal-uniform-load bound ---------------------------------------
    # Both runs share the same ramp-up and ramp-down diagonals, so the time
    # difference between n and n/2 segments is n/2 full diagonals (every
    # layer busy).  A full diagonal advances one segment through the whole
    # model, so S / t_full is the throughput with no ramp at all.
    uniform = None
    if n_seg // 2 >= cfg.n_layers:
        h2 = n_seg // 2
        step_half = lambda: model.armt_forward(tokens[:h2 * cfg.seg_len], h2, hidden, A, z, 0, stream,
                                               B.SCHEDULE_DIAGONAL)
        step_half()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step_half()
        e1.record(stream)
        torch.cuda.synchronize()
        half_ms = e0.elapsed_time(e1)
        t_full = (ms_step - half_ms) / (n_seg - h2)
        uniform = {"ms_per_full_diagonal": t_full,
                   "tokens_per_s": cfg.seg_len / (t_full / 1000.0) if t_full > 0 else None,
                   "ramp_overhead_frac": 1.0 - n_seg * t_full / ms_step,
                   "method": f"(t({n_seg} segments) - t({h2})) / {n_seg - h2} full diagonals"}

    # ---- LM head (tied embedding) over one 8192-token chunk of the output --
    lm = None
    if cfg.dtype == "bf16" and cfg.vocab % 256 == 0:
        r = min(8192, n_tok)
        logits = torch.empty((r, cfg.vocab), dtype=torch.float32, device="cuda")
        model.armt_lm_head(hidden[:r], logits, stream=stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(3):
            model.armt_lm_head(hidden[:r], logits, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        model.armt_sync_status()
        lm_ms = e0.elapsed_time(e1) / 3
        lm = {"rows": r, "vocab": cfg.vocab, "ms": lm_ms,
              "tflops": 2.0 * r * cfg.d_model * cfg.vocab / (lm_ms / 1000.0) / 1e12}
        del logits
        torch.cuda.empty_cache()

    # ---- full-causal-attention LLaMA on the same weights (no memory) -----
    full = None
    if not args.no_full and cfg.dtype == "bf16":
        model.armt_forward_full_attention(tokens, hidden, stream)   # grows its workspace
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        model.armt_forward_full_attention(tokens, hidden, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        model.armt_sync_status()
        full_ms = e0.elapsed_time(e1)
        full = {"ms_per_step": full_ms, "tokens_per_s": n_tok / (full_ms / 1000.0),
                "speedup_diag_over_full": full_ms / ms_step}

    # ---- diagonal batching vs micro-batching (per-segment time) ----------
    # Section 三 of the summary page compares the time per segment of
    # diagonal batching with micro-batching (the sequential schedule run over
    # a batch of B sequences at once).  Same weights; 16 segments per
    # sequence; time per segment of one sequence = t / (segments x B).
    microbatch = None
    if not args.no_microbatch and cfg.dtype == "bf16":
        mb_seg = min(16, n_seg)
        mb_tok = mb_seg * cfg.seg_len
        rng = np.random.default_rng(seed + 1000)
        rows = []
        for sched, bs in ((B.SCHEDULE_SEQUENTIAL, 1), (B.SCHEDULE_SEQUENTIAL, 2), (B.SCHEDULE_SEQUENTIAL, 4),
                          (B.SCHEDULE_SEQUENTIAL, 8), (B.SCHEDULE_SEQUENTIAL, 16),
                          (B.SCHEDULE_DIAGONAL, 1), (B.SCHEDULE_DIAGONAL, 4)):
            tb = torch.from_numpy(rng.integers(0, cfg.vocab, size=(bs, mb_tok)).astype(np.int32)).cuda()
            hb = torch.empty((bs, mb_tok, cfg.d_model), dtype=torch.float32, device="cuda")
            Ab = torch.empty((cfg.n_layers, bs, model.a_elems // cfg.n_layers), dtype=torch.float32, device="cuda")
            zb = torch.empty((cfg.n_layers, bs, model.z_elems // cfg.n_layers), dtype=torch.float32, device="cuda")
            model.armt_forward_batch(tb, hb, Ab, zb, 0, sched, stream)   # sizes the batch workspace
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            model.armt_forward_batch(tb, hb, Ab, zb, 0, sched, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            model.armt_sync_status()
            t_ms = e0.elapsed_time(e1)
            rows.append({"schedule": "diagonal" if sched == B.SCHEDULE_DIAGONAL else "sequential",
                         "batch": bs, "ms": t_ms, "ms_per_segment": t_ms / (mb_seg * bs),
                         "tokens_per_s": bs * mb_tok / (t_ms / 1000.0)})
            del tb, hb, Ab, zb
        microbatch = {"segments_per_sequence": mb_seg, "runs": rows,
                      "batch_workspace_bytes": model.armt_memory_bytes()[1] - ws_create}
        torch.cuda.empty_cache()

    # ---- split precision: activations as bf16 high + low parts -----------
    # The same workload and weights with ARMT_PRECISION_BF16X2: every weight
    # product's K loop runs twice (high, then low part of the activations).
    split = None
    if not args.no_split and cfg.dtype == "bf16" and W is not None:
        cfg_x2 = dataclasses.replace(cfg, precision="bf16x2")
        model_x2 = B.Model(cfg_x2, B.device_weight_tensors(cfg_x2, W))
        torch.cuda.empty_cache()
        model_x2.armt_forward(tokens, n_seg, hidden, A, z, 0, stream, B.SCHEDULE_DIAGONAL)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        model_x2.armt_forward(tokens, n_seg, hidden, A, z, 0, stream, B.SCHEDULE_DIAGONAL)
        e1.record(stream)
        torch.cuda.synchronize()
        model_x2.armt_sync_status()
        x2_ms = e0.elapsed_time(e1)
        split = {"ms_per_step": x2_ms, "tokens_per_s": n_tok / (x2_ms / 1000.0),
                 "slowdown_vs_bf16": x2_ms / ms_step,
                 "workspace_bytes": model_x2.armt_memory_bytes()[1]}
        model_x2.close()
        del model_x2
        torch.cuda.empty_cache()

    # ---- persistent wavefront vs per-diagonal launches (fp32 model) ------
    # The wavefront schedule runs fp32 models: one cooperative launch for the
    # whole forward, each stage of each cell starting when the stages it
    # reads from are done (device-side counters).  A 4-layer d=256 fp32
    # model at 8 and 64 segments of 64 tokens, same weights and tokens.
    wavefront = None
    if not args.no_wavefront:
        cfg_w = dataclasses.replace(I.ARMT_1B, n_layers=4, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                                    ffn_dim=512, vocab=1000, seg_len=64, dtype="f32")
        model_w = B.Model(cfg_w, I.make_weights(cfg_w, 7))
        wavefront = {"workload": "fp32 ARMT, 4 layers, d 256, 4/2 heads of 64, F 512, 64 + 16 rows per cell",
                     "runs": []}
        for n_w in (8, 64):
            tw = torch.from_numpy(I.make_tokens(cfg_w, n_w, 7)).cuda().view(1, -1)
            hw = torch.empty((1, n_w * cfg_w.seg_len, cfg_w.d_model), dtype=torch.float32, device="cuda")
            Aw = torch.empty((cfg_w.n_layers, 1, model_w.a_elems // cfg_w.n_layers), dtype=torch.float32, device="cuda")
            zw = torch.empty((cfg_w.n_layers, 1, model_w.z_elems // cfg_w.n_layers), dtype=torch.float32, device="cuda")
            row = {"segments": n_w}
            for name, sch in (("diagonal", B.SCHEDULE_DIAGONAL), ("wavefront", B.SCHEDULE_WAVEFRONT)):
                model_w.armt_forward_batch(tw, hw, Aw, zw, 0, sch, stream)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(3):
                    model_w.armt_forward_batch(tw, hw, Aw, zw, 0, sch, stream)
                e1.record(stream)
                torch.cuda.synchronize()
                model_w.armt_sync_status()
                row[name + "_ms"] = e0.elapsed_time(e1) / 3
                row[name + "_launches"] = model_w.armt_launch_count(n_w, sch)
            row["speedup_wavefront_over_diagonal"] = row["diagonal_ms"] / row["wavefront_ms"]
            wavefront["runs"].append(row)
        model_w.close()
        del model_w
        torch.cuda.empty_cache()

    # ---- backward pass over reverse diagonals (fp32 model) ----------------
    # armt_backward runs a forward that keeps each cell's inputs and entry
    # state, then the adjoint over the anti-diagonals in reverse (recompute,
    # write, block and read adjoints; all cells of a diagonal per launch).
    # fp32 products on the CUDA cores: the roofline is the fp32 FMA rate,
    # 152 SMs x 128 lanes x 2 FLOP x the sampled SM clock.
    backward = None
    if not args.no_backward:
        small = dataclasses.replace(I.ARMT_1B, n_layers=4, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                                    ffn_dim=512, vocab=1000, seg_len=64, dtype="f32")
        mid = dataclasses.replace(I.ARMT_1B, n_layers=4, d_model=1024, n_q_heads=16, n_kv_heads=4, head_dim=64,
                                  ffn_dim=4096, vocab=4096, seg_len=512, dtype="f32")
        backward = {"workloads": {
            "small": "fp32 ARMT, 4 layers, d 256, 4/2 heads of 64, F 512, 64 + 16 rows per cell",
            "mid": "fp32 ARMT, 4 layers, d 1024, 16/4 heads of 64, F 4096, 512 + 16 rows per cell",
            "main": "the timed model (bf16 forward; fp32 adjoint against fp32 copies of its weights), "
                    "first 8 segments"},
            "runs": []}
        legs = [("small", small, 8), ("small", small, 64), ("mid", mid, 8)]
        if cfg.n_layers * cfg.d_model <= 16 * 2048:  # the main model when it is ARMT-1B-sized or smaller
            legs.append(("main", cfg, min(8, n_seg)))
        for wl, cfg_b, n_b in legs:
            own = wl != "main"
            model_b = B.Model(cfg_b, I.make_weights(cfg_b, 8)) if own else model
            tb = (torch.from_numpy(I.make_tokens(cfg_b, n_b, 8)) if own
                  else torch.from_numpy(tok_np[:n_b * cfg.seg_len].copy())).cuda()
            rng_b = torch.Generator(device="cuda")
            rng_b.manual_seed(8)
            cot_h = torch.randn((tb.numel(), cfg_b.d_model), generator=rng_b, device="cuda")
            model_b.backward(tb, cot_hidden=cot_h)           # sizes the workspace
            hb = torch.empty((1, tb.numel(), cfg_b.d_model), dtype=torch.float32, device="cuda")
            Ab = torch.empty((cfg_b.n_layers, 1, model_b.a_elems // cfg_b.n_layers), dtype=torch.float32,
                             device="cuda")
            zb = torch.empty((cfg_b.n_layers, 1, model_b.z_elems // cfg_b.n_layers), dtype=torch.float32,
                             device="cuda")
            shapes_b = I.weight_shapes(cfg_b)
            grads_b = {k: torch.empty(shapes_b[k], dtype=torch.float32, device="cuda") for k in shapes_b}
            row = {"workload": wl, "segments": n_b, "tokens": tb.numel()}
            torch.cuda.nvtx.range_push(f"backward:{wl}:{n_b}")  # lets a profiler pick one leg
            for name in ("forward", "backward"):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                for _ in range(3):
                    if name == "forward":
                        model_b.armt_forward_batch(tb.view(1, -1), hb, Ab, zb, 0, B.SCHEDULE_DIAGONAL, stream)
                    else:
                        model_b.armt_backward(tb, grads_b, cot_hidden=cot_h, stream=stream)
                e1.record(stream)
                torch.cuda.synchronize()
                model_b.armt_sync_status()
                row[name + "_ms"] = e0.elapsed_time(e1) / 3
            torch.cuda.nvtx.range_pop()
            launches_b, flops_b, ws_b = model_b.armt_backward_stats()
            adj_ms = row["backward_ms"] - row["forward_ms"]
            row.update({"backward_includes_forward": True, "adjoint_ms": adj_ms,
                        "adjoint_launches": launches_b, "adjoint_gflop": flops_b / 1e9,
                        "adjoint_tflops": flops_b / (adj_ms * 1e-3) / 1e12,
                        "tokens_per_s": tb.numel() / (row["backward_ms"] * 1e-3),
                        "workspace_bytes": ws_b})
            backward["runs"].append(row)
            if own:
                model_b.close()
            del model_b, grads_b
            torch.cuda.empty_cache()
        # fp32 FMA peak from the unit counts and the SM clock sampled in the timed region
        mhz = (clocks or {}).get("sm_mhz") or 2070.0
        backward["fp32_fma_peak_tflops"] = 152 * 128 * 2 * mhz * 1e6 / 1e12
        for row in backward["runs"]:
            row["adjoint_frac_of_fp32_peak"] = row["adjoint_tflops"] / backward["fp32_fma_peak_tflops"]

    # ---- end to end through the host-buffer entry point ------------------
    e2e = None
    if not args.no_e2e:
        h_tok = torch.from_numpy(tok_np).pin_memory()
        h_hidden = torch.empty((n_tok, cfg.d_model), dtype=torch.float32).pin_memory()
        h_A = torch.empty(model.a_elems, dtype=torch.float32).pin_memory()
        h_z = torch.empty(model.z_elems, dtype=torch.float32).pin_memory()
        model.armt_forward_host(h_tok, n_seg, h_hidden, h_A, h_z, 0, B.SCHEDULE_DIAGONAL, stream)
        # the same K steps as the headline; host wall clock, because every
        # call synchronises (its copies back to the host are part of the step)
        t0 = time.perf_counter()
        ke = args.steps
        for _ in range(ke):
            model.armt_forward_host(h_tok, n_seg, h_hidden, h_A, h_z, 0, B.SCHEDULE_DIAGONAL, stream)
        dt = (time.perf_counter() - t0) / ke
        e2e = {"value": world * n_tok / dt, "unit": UNIT, "h2d_bytes_per_step": int(h_tok.numel() * 4),
               "d2h_bytes_per_step": int((h_hidden.numel() + h_A.numel() + h_z.numel()) * 4), "steps": ke}

    # ---- oracle on the host cores (rank 0, N=1 only) ---------------------
    cpu = None
    if not args.no_cpu and rank == 0 and world == 1 and W is not None:
        t = oracle_sample_seconds(cfg, W, tok_np)
        cpu = {"value": cfg.seg_len / t, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 oracle, segment 0 ({cfg.seg_len} tokens) through all {cfg.n_layers} "
                         f"layers ({t:.1f} s); per-segment cost is constant in the segment recurrence"}

    # ---- device memory: recurrent state vs a full-attention KV cache -----
    w_bytes, _, fw_bytes = model.armt_memory_bytes()
    ws_bytes = ws_create
    state_bytes = (model.a_elems + model.z_elems) * 4
    kv_bytes = 2 * cfg.n_layers * n_tok * cfg.n_kv_heads * cfg.head_dim * 2
    memory = {"weights_bytes": w_bytes, "armt_workspace_bytes": ws_bytes,
              "armt_state_bytes": state_bytes, "full_attention_workspace_bytes": fw_bytes or None,
              "kv_cache_bytes_full_llama": kv_bytes,
              "kv_cache_over_armt_state": kv_bytes / state_bytes,
              "note": "ARMT workspace is fixed at create (one activation slot per layer) and its "
                      "state is O(L d P) whatever the length; a full-attention model holds a bf16 "
                      "KV cache of 2 L T Hkv hd entries at context T"}

    launches = model.armt_launch_count(n_seg, B.SCHEDULE_DIAGONAL) * args.steps
    if rank == 0:
        out = {
            "metric": metric_name(args.workload), "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": args.workload, "tokens": n_tok, "segments": n_seg,
                       "segment_len": cfg.seg_len, "memory_tokens": cfg.n_mem, "layers": cfg.n_layers,
                       "batch": 1, "schedule": "diagonal", "parallelism": "replicas" if world > 1 else "single",
                       "precision": "bf16 weight-product operands, fp16 attention operands, fp32 accumulation",
                       "l2": "no flush: every diagonal re-reads all layers' weights (~2 GB) and "
                             "~1 GB of activations, far above the 129 MB L2"},
            "roofline": {"bound": "tensor", "kernel": "grouped GEMM gate-up + SwiGLU (tcgen05)",
                         "achieved": gu_tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": (gu_tflops / peak) if gu_tflops else None, "traffic": gu_traffic,
                         "traffic_unit": "bytes per launch (ncu dram__bytes_read+write, scaled by cells)",
                         "peak_source": f"bf16_tflops_sustained ({peak_src})",
                         "all_gemms_tflops": gemm_tflops,
                         "all_gemms_note": "from one extra forward with every launch timed (after the timed region)",
                         "all_gemms_frac": (gemm_tflops / peak) if gemm_tflops else None},
            "model_tflops": total_flops * args.steps / (ms_total / 1000.0) / 1e12,
            "kernels": per_class,
            "sequential": seq,
            "uniform_bound": uniform,
            "lm_head": lm,
            "full_attention": full,
            "microbatch": microbatch,
            "split_precision": split,
            "wavefront": wavefront,
            "backward": backward,
            "memory": memory,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": int(launches),
            "clocks": clocks,
        }
        print(json.dumps(out), flush=True)
    model.close()
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
