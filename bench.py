"""Benchmark of the Simple GLA mixer hot path on GB300.

One step = the whole hot path on its two workloads:
  * chunked forward + backward at the training shape B=32, T=2048, H=16, dk=96, dv=192
    (bf16 inputs, fp32 outputs; the forward saves the gate sigmoid(q.(a*k)) and the backward
    reads it, as a training step keeps its saved activations) -- `value` is its throughput in
    tokens/s;
  * one recurrent decode step over the serving pool of 1,280 sequences x 24 layers x 16
    heads of 96x192 fp32 states (36.2 GB resident in HBM) -- reported in `decode` as GB/s.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle instead (the
reference arm: the plain definition, on the host cores, one bounded sample per step).

Inputs are synthetic (seeded Gaussians with the workloads' shapes and scales) and larger
than L2, so no flush is needed between timed iterations.  Kernel times come from CUDA
events on the launching stream; SM clocks are sampled with nvidia-smi during the timed
region.  Multi-GPU (torchrun): every rank runs the same per-GPU workload (independent
replicas, no collective on the data path); times are maxed over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GLA fwd+bwd tokens/s (H=16,T=2048) and decode-step GB/s vs HBM roofline"
B, T, H, DK, DV = 32, 2048, 16, 96, 192
N_SEQ, N_LAYERS = 1280, 24
def workload_name(b: int = B, n_seq: int = N_SEQ) -> str:
    return (f"GLA chunked fwd+bwd B={b} T=2048 H=16 dk=96 dv=192 chunk=128 bf16-in/fp32-out, "
            f"plus one decode step over {n_seq} seqs x 24 layers x 16 heads of 96x192 fp32 states")


WORKLOAD = workload_name()
# Algorithmic work per unit (what the calls must move / compute at minimum)
# the training step saves the gate sigmoid(z) (fp32 per token-head) in the forward for the backward
# and the state copies (36,864 B fp16 + a 4-byte exponent per chunk of 128 tokens, 288.03 B per
# token-head), written by the forward and read by the backward's dq part
FWD_BYTES_TH = (96 + 96 + 192) * 2 + 192 * 4 + 4         # bf16 q,k,v in, fp32 o, gate out = 1540
BWD_BYTES_TH = (96 + 96 + 192 + 192) * 2 + 4 + (96 + 96 + 192) * 4  # + dO, gate in; dq,dk,dv = 2692
SAVED_BYTES_TH = (96 * 192 * 2 + 4) / 128                 # state copies: 288.03
FWD_FLOPS_TH = 2 * (128 * 96 + 128 * 192 + 96 * 192 + 96 * 192)  # QK^T, PV, QS, K^T V = 147456
BWD_FLOPS_TH = 319488                                     # 9 dense chunk matmuls per token-head
DEC_BYTES_STATE = 2 * 96 * 192 * 4 + (96 + 96 + 192 + 192) * 4  # state r+w, q,k,v,o = 149760


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="of measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="of fallback")


def traffic_record(kernel: str):
    """dram bytes per unit from an ncu capture (profiles/traffic.json), if the kernel
    source it was taken on is unchanged; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    m = hashlib.sha256()
    for f in rec["source"]:
        src = os.path.join(ROOT, "gated_linear_attention_chunked_gb300", "csrc", f)
        if not os.path.exists(src):
            return None
        m.update(open(src, "rb").read())
    return rec if m.hexdigest()[:16] == rec.get("source_sha256_16") else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open(os.devnull, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                txt, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                txt, _ = self.proc.communicate()
            self.lines = [l for l in txt.splitlines() if l.strip()]
        if self.out:
            self.out.close()

    def mark(self, which: str):
        setattr(self, which, time.time())

    def summary(self):
        import datetime
        import statistics
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t_start", None), getattr(self, "t_end", None)
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if t0 is not None and not (t0 <= ts <= t1):
                    continue  # outside the timed region
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


# --------------------------------------------------------------------------- CPU oracle
def oracle_sample(n_seq: int, seed: int = 2):
    """Time the fp64 oracle's fwd+bwd over `n_seq` sequences of the training workload."""
    import numpy as np

    import oracle
    import synth
    x = synth.chunk_inputs("train_fwd_bwd", B=n_seq)
    g = oracle.decay_schedule(H).astype(np.float32).astype(np.float64)
    t0 = time.perf_counter()
    oracle.fwd(x["q"], x["k"], x["v"], g, x["a"])
    oracle.bwd(x["q"], x["k"], x["v"], g, x["a"], x["dO"])
    dt = time.perf_counter() - t0
    return n_seq * T / dt, dt


def oracle_decode_sample(every: int = 64, steps: int = 40, seed: int = 3):
    """Time the fp64 oracle's decode step over every `every`-th sequence of the serving pool
    (all 24 layers x 16 heads each); returns (states per second, states, seconds)."""
    import numpy as np

    import oracle
    import synth
    n = len(range(0, N_SEQ, every))
    rng = np.random.default_rng(seed)
    st = rng.standard_normal((n, N_LAYERS, H, DK, DV)) * 0.5
    q, k, v = synth.decode_token(seed, n, N_LAYERS, H)
    a = synth.aug_balance(seed, (N_LAYERS, H, DK), 0.02)
    g = oracle.decay_schedule(H).astype(np.float32).astype(np.float64)
    oracle.decode_step(st, q, k, v, g, a)  # warm-up (page-in, thread start)
    t0 = time.perf_counter()
    for _ in range(steps):
        _, st = oracle.decode_step(st, q, k, v, g, a)
    dt = time.perf_counter() - t0
    n_states = n * N_LAYERS * H
    return n_states * steps / dt, n_states, dt


def oracle_long_prefill_sample(t_sample: int = 65536, seed: int = 4):
    """Time the fp64 oracle's forward over the first `t_sample` tokens of both long-prefill
    sequences (B=2, H=16, with the initial state); returns (tokens per second, seconds)."""
    import numpy as np

    import oracle
    import synth
    x = synth.chunk_inputs("long_prefill", T=t_sample)
    g = oracle.decay_schedule(H).astype(np.float32).astype(np.float64)
    t0 = time.perf_counter()
    oracle.fwd(x["q"], x["k"], x["v"], g, x["a"], x["init_state"])
    dt = time.perf_counter() - t0
    return 2 * t_sample / dt, dt


def reduce_max(values, dist, device):
    """Element-wise max over ranks of this rank's values (timings): the slowest rank sets the
    job's time.  dist None = one process."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_rate(world, units_per_rank, seconds):
    """Whole-job throughput: the units every rank processed over the (max-over-ranks) time."""
    return world * units_per_rank / seconds


def run_cpu_configs(args):
    """--cpu-configs: the fp64 oracle timed on this host's cores on every workload -- tiny
    fp32 fwd+bwd (whole), the layer forward B=8 (whole), the training fwd+bwd B=32 (whole),
    the decode step (every 64th sequence of the pool, extrapolated) and the long prefill
    (whole: both sequences of 131072 tokens).  One JSON line; the CPU baseline the GPU numbers
    are reported beside."""
    import numpy as np

    import oracle
    import synth
    cores = os.cpu_count() or 1
    try:
        import platform
        cpu = platform.processor() or platform.machine()
    except Exception:  # noqa: BLE001 - informational only
        cpu = "unknown"
    out = dict(part="cpu_configs", cores=cores, cpu=cpu, unit_note="tokens/s unless stated")

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    x = synth.chunk_inputs("tiny_fp32")
    g2 = oracle.decay_schedule(2).astype(np.float32).astype(np.float64)
    dt = timed(lambda: (oracle.fwd(x["q"], x["k"], x["v"], g2, x["a"]),
                        oracle.bwd(x["q"], x["k"], x["v"], g2, x["a"], x["dO"])))
    out["tiny_fp32_fwd_bwd"] = dict(s=dt, tokens_per_s=256 / dt)
    g = oracle.decay_schedule(H).astype(np.float32).astype(np.float64)
    x = synth.chunk_inputs("layer_fwd_aug")
    dt = timed(lambda: oracle.fwd(x["q"], x["k"], x["v"], g, x["a"]))
    out["layer_fwd_B8"] = dict(s=dt, tokens_per_s=8 * T / dt)
    rate, dt = oracle_sample(32)
    out["train_fwd_bwd_B32"] = dict(s=dt, tokens_per_s=rate)
    st_rate, n_st, dt = oracle_decode_sample()
    out["decode_pool"] = dict(s=dt, states=n_st, steps=40, gbs=st_rate * DEC_BYTES_STATE / 1e9,
                              ms_per_step_extrapolated=1e3 * N_SEQ * N_LAYERS * H / st_rate)
    rate, dt = oracle_long_prefill_sample(t_sample=131072)
    out["long_prefill_fwd"] = dict(s=dt, tokens=2 * 131072, tokens_per_s=rate)
    print(json.dumps(out), flush=True)
    return 0


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    import numpy as np
    for _ in range(args.warmup):
        oracle_sample(1)
    rates, times = [], []
    for _ in range(args.steps):
        r, dt = oracle_sample(1)
        rates.append(r)
        times.append(dt)
    tot_tok = args.steps * T
    value = tot_tok / sum(times)
    line = dict(
        impl="reference", metric=METRIC, value=value, unit="tokens/s", n_gpus=args.gpus,
        steps=args.steps, warmup=args.warmup, ms_per_step=1e3 * float(np.mean(times)),
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
        data="synthetic (seeded Gaussians, training-shape recipe)",
        config=dict(workload=WORKLOAD, B=B, T=T, H=H, dk=DK, dv=DV, chunk=128,
                    step_sample="oracle fwd+bwd over 1 of the 32 sequences (T=2048, H=16)"),
        cpu_baseline=dict(value=value, unit="tokens/s", cores=cores, kind="oracle",
                          sample="fp64 token-by-token fwd + hand-derived bwd, 1 sequence x "
                                 "T=2048 x H=16 per step, threaded over heads"),
        e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0),
    )
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch

    Bn, Ns = args.batch, args.n_seq
    do_fwd = args.part in ("all", "fwd")
    do_bwd = args.part in ("all", "bwd")
    do_dec = args.part in ("all", "decode")

    import gated_linear_attention_chunked_gb300 as gla
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    gla.load()
    gla.set_pass_overlap(args.pass_overlap)
    gla.set_split_parts(args.split_parts)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pk = peaks()
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)

    def randn(*shape, std=1.0, dtype=torch.float32):
        return (torch.randn(*shape, generator=gen, device=dev) * std).to(dtype)

    # ---- training-shape tensors (bf16 inputs, fp32 outputs), resident in HBM
    gam = gla.decay_schedule(H).to(dev)
    a = randn(H, DK, std=0.02)
    if do_fwd or do_bwd:
        q = randn(Bn, T, H, DK, std=DK ** -0.5, dtype=torch.bfloat16)
        k = randn(Bn, T, H, DK, dtype=torch.bfloat16)
        v = randn(Bn, T, H, DV, dtype=torch.bfloat16)
        dO = randn(Bn, T, H, DV, dtype=torch.bfloat16)
        o = torch.empty(Bn, T, H, DV, device=dev)
        fin = torch.empty(Bn, H, DK, DV, device=dev)
        gate = torch.empty(Bn, H, T, device=dev)  # sigmoid(z), saved by the forward
        saved = (torch.empty(gla.chunk_saved_states_size(Bn, T, H), dtype=torch.uint8, device=dev)
                 if args.saved_states else None)  # the state copies, saved by the forward
        ws = torch.empty(max(1, gla.chunk_bwd_workspace_size(Bn, T, H, gla.GLA_BF16)),
                         dtype=torch.uint8, device=dev)
        # a backward alone reads what this forward saves
        gla.chunk_fwd(q, k, v, gam, a, out=o, final_state=fin, gate=gate, saved_states=saved)

    # ---- serving pool: 1280 x 24 x 16 states, warmed by 64 recurrent steps from zero
    if do_dec:
        st = torch.zeros(Ns, N_LAYERS, H, DK, DV, device=dev)
        ad = randn(N_LAYERS, H, DK, std=0.02)
        dq_ = randn(Ns, N_LAYERS, H, DK, std=DK ** -0.5)
        dk_ = randn(Ns, N_LAYERS, H, DK)
        dv_ = randn(Ns, N_LAYERS, H, DV)
        od = torch.empty(Ns, N_LAYERS, H, DV, device=dev)
        for _ in range(64):
            dq_.normal_(0.0, DK ** -0.5, generator=gen)
            dk_.normal_(generator=gen)
            dv_.normal_(generator=gen)
            gla.decode_step(st, dq_, dk_, dv_, gam, ad, out=od)
        dq_.normal_(0.0, DK ** -0.5, generator=gen)
        dk_.normal_(generator=gen)
        dv_.normal_(generator=gen)
    torch.cuda.synchronize()
    if gla.get_device_error() != 0:
        raise RuntimeError("device error during setup")

    stream = torch.cuda.current_stream()
    n_states = Ns * N_LAYERS * H

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        if do_fwd:
            gla.chunk_fwd(q, k, v, gam, a, out=o, final_state=fin, gate=gate, saved_states=saved)
        if evs:
            evs[1].record(stream)
        if do_bwd:
            gla.chunk_bwd(q, k, v, gam, a, dO, gate=gate, saved_states=saved, workspace=ws)
        if evs:
            evs[2].record(stream)
        if do_dec:
            gla.decode_step(st, dq_, dk_, dv_, gam, ad, out=od)
        if evs:
            evs[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        time.sleep(0.5)  # let the sampler come up
        clk.mark("t_start")
        t_wall = time.perf_counter()
        for s in range(args.steps):
            step(evs[s])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        clk.mark("t_end")
    if dist:
        dist.barrier()
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    dec_ms = [e[2].elapsed_time(e[3]) for e in evs]
    tot_ms = [e[0].elapsed_time(e[3]) for e in evs]
    if gla.get_device_error() != 0:
        raise RuntimeError("device error in the timed region")
    sums = reduce_max([sum(fwd_ms), sum(bwd_ms), sum(dec_ms), sum(tot_ms)], dist, dev)
    fwd_t, bwd_t, dec_t, tot_t = (x / args.steps for x in sums)  # ms per step
    if args.part != "all":
        part_ms = dict(fwd=fwd_t, bwd=bwd_t, decode=dec_t)[args.part]
        if rank == 0:
            print(json.dumps(dict(part=args.part, ms=part_ms, batch=Bn, n_seq=Ns, steps=args.steps,
                                  warmup=args.warmup, clocks=clk.summary())), flush=True)
        if dist:
            dist.destroy_process_group()
        return 0
    tokens = Bn * T  # the batch actually run (32 unless --batch says otherwise)
    value = job_rate(world, tokens, (fwd_t + bwd_t) * 1e-3)
    dec_bytes = n_states * DEC_BYTES_STATE
    dec_gbs = dec_bytes / (dec_t * 1e-3) / 1e9
    th = Bn * T * H
    # our kernels per step: chunk fwd, chunk bwd, d_aug reduction, decode, and the two segment
    # passes of each chunked call whose plan cuts pairs into parts
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    # segment passes of a cut call: the sum pass, and the link pass unless there are two parts
    parts_f = gla.split_plan(Bn, T, H, False, n_sm)[1]
    parts_b = gla.split_plan(Bn, T, H, 2 if args.saved_states else 1, n_sm)[1]
    pass_f = 0 if parts_f <= 1 else (1 if parts_f == 2 else 2)
    pass_b = 0 if parts_b <= 1 else (1 if parts_b == 2 else 2)
    gpu_launches_per_step = 4 + pass_f + pass_b

    def roof(bound, achieved, peak, unit, traffic):
        return dict(bound=bound, achieved=achieved, peak=peak, unit=unit, frac=achieved / peak,
                    traffic=traffic, peak_source=pk["src"])

    tr_dec = traffic_record("decode")
    tr_fwd = traffic_record("chunk_fwd")
    tr_bwd = traffic_record("chunk_bwd")
    roofline = roof("hbm", dec_gbs, pk["hbm"], "GB/s",
                    None if tr_dec is None else tr_dec["bytes_per_unit"] * n_states)
    roofline["kernel"] = "decode_kernel (dominant: largest share of the step time)"
    fb_th = FWD_BYTES_TH + (SAVED_BYTES_TH if args.saved_states else 0.0)
    bb_th = BWD_BYTES_TH + (SAVED_BYTES_TH if args.saved_states else 0.0)
    fwd_gbs = th * fb_th / (fwd_t * 1e-3) / 1e9
    bwd_gbs = th * bb_th / (bwd_t * 1e-3) / 1e9
    roof_fwd = roof("hbm", fwd_gbs, pk["hbm"], "GB/s",
                    None if tr_fwd is None else tr_fwd["bytes_per_unit"] * th)
    roof_fwd["tensor"] = dict(achieved=th * FWD_FLOPS_TH / (fwd_t * 1e-3) / 1e12, peak=pk["bf16"],
                              unit="TFLOP/s", frac=th * FWD_FLOPS_TH / (fwd_t * 1e-3) / 1e12 / pk["bf16"])
    roof_bwd = roof("hbm", bwd_gbs, pk["hbm"], "GB/s",
                    None if tr_bwd is None else tr_bwd["bytes_per_unit"] * th)
    roof_bwd["tensor"] = dict(achieved=th * BWD_FLOPS_TH / (bwd_t * 1e-3) / 1e12, peak=pk["bf16"],
                              unit="TFLOP/s", frac=th * BWD_FLOPS_TH / (bwd_t * 1e-3) / 1e12 / pk["bf16"])

    # each chunk call alone: the same call 20 times back to back after the step loop (CUDA
    # events on the launching stream; inputs > L2), next to its time inside the step above
    def alone_ms(fn, n=20):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return reduce_max([e0.elapsed_time(e1) / n], dist, dev)[0]

    for roof_, ms_, by_ in (
            (roof_fwd, alone_ms(lambda: gla.chunk_fwd(q, k, v, gam, a, out=o, final_state=fin,
                                                      gate=gate, saved_states=saved)), fb_th),
            (roof_bwd, alone_ms(lambda: gla.chunk_bwd(q, k, v, gam, a, dO, gate=gate,
                                                      saved_states=saved, workspace=ws)), bb_th)):
        roof_["alone"] = dict(ms=ms_, achieved=th * by_ / (ms_ * 1e-3) / 1e9, unit="GB/s",
                              frac=th * by_ / (ms_ * 1e-3) / 1e9 / pk["hbm"],
                              note="the same call 20 times back to back after the step loop; "
                                   "the fields above are its time inside the step")
    if gla.get_device_error() != 0:
        raise RuntimeError("device error in the chunk calls timed alone")

    # ---- end to end through the public API: pinned host inputs -> HBM -> fwd+bwd -> d_aug.
    # Every step copies its own inputs from pinned host memory and reads its d_aug back; as
    # in a training loop's prefetch, the copy of step s+1 runs on a second stream into the
    # other of two device buffers while step s computes (host->device is ~5.8 ms per step
    # here, the kernels ~2 ms).  The clock starts before the first copy and stops after the
    # last read-back has landed.
    e2e = e2e_full_readback = None
    if not args.no_e2e:
        hq, hk, hv, hdO = (x.cpu().pin_memory() for x in (q, k, v, dO))
        e2e_steps = max(3, min(args.steps, 10))
        h_daug = torch.empty(e2e_steps, H, DK).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdO))
        d2h = H * DK * 4
        bufs = [tuple(torch.empty_like(x) for x in (q, k, v, dO)) for _ in range(2)]
        copy_stream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]

        def e2e_run(nsteps):
            for s_ in range(nsteps):
                i = s_ % 2
                with torch.cuda.stream(copy_stream):
                    if s_ >= 2:
                        copy_stream.wait_event(consumed[i])  # step s-2 is done with buffer i
                    for d, hsrc in zip(bufs[i], (hq, hk, hv, hdO)):
                        d.copy_(hsrc, non_blocking=True)
                    copied[i].record(copy_stream)
                stream.wait_event(copied[i])
                bq, bk, bv, bdO = bufs[i]
                gla.chunk_fwd(bq, bk, bv, gam, a, out=o, final_state=fin, gate=gate,
                              saved_states=saved)
                _, _, _, daug, _ = gla.chunk_bwd(bq, bk, bv, gam, a, bdO, gate=gate,
                                                 saved_states=saved, workspace=ws,
                                                 want_d_init_state=False)
                consumed[i].record(stream)
                h_daug[s_].copy_(daug, non_blocking=True)
            torch.cuda.synchronize()

        def windows(run):
            """three timed windows of e2e_steps steps each (barrier + sync around each, max over
            ranks): the host link is shared with the machine's other GPUs, so one window can
            catch another job's transfer; the median is reported and all three listed"""
            ts = []
            for _ in range(3):
                if dist:
                    dist.barrier()
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                run(e2e_steps)
                ts.append(reduce_max([time.perf_counter() - t0], dist, dev)[0])
            return sorted(ts)[1], ts

        e2e_run(2)  # warm-up
        tt, tt_all = windows(e2e_run)
        e2e = dict(value=job_rate(world, tokens * e2e_steps, tt), unit="tokens/s",
                   h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                   windows_s=tt_all, steps_per_window=e2e_steps,
                   path="pinned host q,k,v,dO -> gla chunk_fwd + chunk_bwd -> host d_aug. "
                        "Returned to the host: d_aug, the step's parameter gradient (the "
                        "mixer's only trained parameter; the decay is fixed) -- the scalar-"
                        "like result a training step reads back; o and dq, dk, dv feed "
                        "device-side projections and stay in HBM (e2e_full_readback copies "
                        "them back too). Next step's inputs copied on a second stream during "
                        "this step's kernels (two device buffers)")

        # the same loop with every output copied back to pinned host memory each step: o,
        # dq, dk, dv and d_aug (the device->host copy of step s runs on a third stream while
        # step s+1 computes; its outputs go to the other of two device buffers)
        outs = [dict(o=torch.empty_like(o)) for _ in range(2)]
        shapes = dict(o=(Bn, T, H, DV), dq=(Bn, T, H, DK), dk=(Bn, T, H, DK), dv=(Bn, T, H, DV))
        h_out = {n_: torch.empty(sh, dtype=torch.float32).pin_memory() for n_, sh in shapes.items()}
        d2h_full = sum(x.numel() * 4 for x in h_out.values()) + H * DK * 4
        back_stream = torch.cuda.Stream(device=dev)
        computed = [torch.cuda.Event() for _ in range(2)]
        read = [torch.cuda.Event() for _ in range(2)]
        ws_full = torch.empty(max(1, gla.chunk_bwd_workspace_size(Bn, T, H, gla.GLA_BF16)),
                              dtype=torch.uint8, device=dev)

        def e2e_full(nsteps):
            for s_ in range(nsteps):
                i = s_ % 2
                with torch.cuda.stream(copy_stream):
                    if s_ >= 2:
                        copy_stream.wait_event(consumed[i])
                    for d, hsrc in zip(bufs[i], (hq, hk, hv, hdO)):
                        d.copy_(hsrc, non_blocking=True)
                    copied[i].record(copy_stream)
                stream.wait_event(copied[i])
                if s_ >= 2:
                    stream.wait_event(read[i])  # step s-2's outputs have left buffer i
                bq, bk, bv, bdO = bufs[i]
                ob = outs[i]
                gla.chunk_fwd(bq, bk, bv, gam, a, out=ob["o"], final_state=fin, gate=gate,
                              saved_states=saved)
                dq_, dk_, dv_, daug, _ = gla.chunk_bwd(bq, bk, bv, gam, a, bdO, gate=gate,
                                                       saved_states=saved, workspace=ws_full,
                                                       want_d_init_state=False)
                consumed[i].record(stream)
                ob["dq"], ob["dk"], ob["dv"] = dq_, dk_, dv_
                for x_ in (dq_, dk_, dv_, daug):  # read on back_stream: keep until it has
                    x_.record_stream(back_stream)
                computed[i].record(stream)
                with torch.cuda.stream(back_stream):
                    back_stream.wait_event(computed[i])
                    for n_ in ("o", "dq", "dk", "dv"):
                        h_out[n_].copy_(ob[n_], non_blocking=True)
                    h_daug[s_ % e2e_steps].copy_(daug, non_blocking=True)
                    read[i].record(back_stream)
            torch.cuda.synchronize()

        e2e_full(2)  # warm-up
        tf_, tf_all = windows(e2e_full)
        e2e_full_readback = dict(
            value=job_rate(world, tokens * e2e_steps, tf_), unit="tokens/s",
            h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h_full,
            windows_s=tf_all, steps_per_window=e2e_steps,
            path="pinned host q,k,v,dO -> gla chunk_fwd + chunk_bwd -> pinned host o, dq, dk, "
                 "dv, d_aug every step (device->host on a third stream, overlapping the next "
                 "step; bound by the host link)")

        # the host link alone: the same copies with nothing else running (best of 3), so that
        # each e2e figure can be read against the rate the link gives here
        def link_ms(pairs):
            best = float("inf")
            for _ in range(3):
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(copy_stream):
                    e0.record(copy_stream)
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
                    e1.record(copy_stream)
                e1.synchronize()
                best = min(best, e0.elapsed_time(e1))
            return best

        h2d_ms = link_ms(list(zip(bufs[0], (hq, hk, hv, hdO))))
        d2h_ms = link_ms([(h_out[n_], outs[0][n_]) for n_ in ("o", "dq", "dk", "dv")])
        h2d_gbs, d2h_gbs = h2d / h2d_ms / 1e6, (d2h_full - d2h) / d2h_ms / 1e6
        e2e_ms, full_ms = 1e3 * tt / e2e_steps, 1e3 * tf_ / e2e_steps
        e2e["link"] = dict(h2d_gbs=h2d_gbs, bound_ms=h2d_ms, ms_per_step=e2e_ms,
                           frac=h2d_ms / e2e_ms,
                           note="host->device copy of the step's inputs alone (best of 3); "
                                "frac = that time / the e2e time per step")
        bound_full = max(h2d_ms, d2h_ms)
        e2e_full_readback["link"] = dict(h2d_gbs=h2d_gbs, d2h_gbs=d2h_gbs, bound_ms=bound_full,
                                         ms_per_step=full_ms, frac=bound_full / full_ms,
                                         note="the slower direction's copies alone (best of 3); "
                                              "frac = that time / the e2e time per step")
        del bufs, outs

    cpu = cpu_dec = cpu_long = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        rate, dt = oracle_sample(args.cpu_seqs)
        cpu = dict(value=rate, unit="tokens/s", cores=cores, kind="oracle",
                   sample=f"fp64 oracle fwd+bwd over {args.cpu_seqs} of the 32 sequences "
                          f"(T=2048, H=16) = {args.cpu_seqs * T} tokens, {dt:.1f} s")
        st_rate, n_st, dtd = oracle_decode_sample()
        cpu_dec = dict(value=st_rate * DEC_BYTES_STATE / 1e9, unit="GB/s", cores=cores,
                       kind="oracle", states_per_s=st_rate,
                       ms_per_step_extrapolated=1e3 * n_states / st_rate,
                       sample=f"fp64 oracle decode step over every 64th sequence of the pool "
                              f"({n_st} states: 20 sequences x 24 layers x 16 heads), 40 steps, "
                              f"{dtd:.1f} s; GB/s counts the same algorithmic bytes as the GPU "
                              f"line; ms_per_step_extrapolated = the whole 1280-sequence pool at "
                              f"this rate (linear extrapolation)")
        lp_rate, dtl = oracle_long_prefill_sample()
        cpu_long = dict(value=lp_rate, unit="tokens/s", cores=cores, kind="oracle",
                        sample=f"fp64 oracle forward over the first 65536 of the 131072 tokens of "
                               f"both long-prefill sequences (H=16, initial state), {dtl:.1f} s")

    clocks = clk.summary()
    line = dict(
        metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=tot_t, higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype="f16-mma/f32-acc (bf16 in, fp32 out); decode f32",
        data="synthetic (seeded Gaussians with the workloads' shapes and scales)",
        config=dict(workload=workload_name(Bn, Ns), B=Bn, T=T, H=H, dk=DK, dv=DV, chunk=128,
                    decode_pool=[Ns, N_LAYERS, H, DK, DV], parallelism=f"replicas x{world}",
                    l2="inputs larger than L2 (1.2 GB chunk inputs, 36 GB state pool); no flush"),
        roofline=roofline,
        decode=dict(value=dec_gbs, unit="GB/s", ms_per_step=dec_t, states=n_states,
                    frac_of_hbm=dec_gbs / pk["hbm"], peak_source=pk["src"]),
        parts_ms=dict(chunk_fwd=fwd_t, chunk_bwd=bwd_t, decode=dec_t),
        roofline_chunk_fwd=roof_fwd, roofline_chunk_bwd=roof_bwd,
        cpu_baseline=cpu, cpu_baseline_decode=cpu_dec, cpu_baseline_long_prefill=cpu_long,
        e2e=e2e, e2e_full_readback=e2e_full_readback,
        gpu_launches=gpu_launches_per_step * args.steps,
        gpu_launches_detail="per step: chunk fwd, chunk bwd, d_aug reduction, decode"
                            + (f", fwd segment passes ({pass_f})" if pass_f else "")
                            + (f", bwd segment passes ({pass_b})" if pass_b else ""),
        clocks=clocks, wall_s_timed=t_wall,
    )
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def run_fused(args):
    """--part fused: the forward followed by the standalone output epilogue, against the
    forward with the epilogue fused in (y only, and y + o), at the training shape."""
    import torch
    import gated_linear_attention_chunked_gb300 as gla
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gla.load()
    Bf, tiers = args.batch, 4
    gen = torch.Generator(device=dev)
    gen.manual_seed(31)
    q = (torch.randn(Bf, T, H, DK, generator=gen, device=dev) * DK ** -0.5).bfloat16()
    k = torch.randn(Bf, T, H, DK, generator=gen, device=dev).bfloat16()
    v = torch.randn(Bf, T, H, DV, generator=gen, device=dev).bfloat16()
    g = torch.randn(Bf, T, H, DV, generator=gen, device=dev).bfloat16()
    a = 0.02 * torch.randn(H, DK, generator=gen, device=dev)
    w = 1.0 + 0.2 * torch.randn(tiers, DV, generator=gen, device=dev)
    gam = gla.decay_schedule(H).to(dev)
    o = torch.empty(Bf, T, H, DV, device=dev)
    y = torch.empty_like(o)
    stream = torch.cuda.current_stream()

    def timed(fn, n):
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def separate():
        gla.chunk_fwd(q, k, v, gam, a, out=o, want_final_state=False)
        gla.head_norm_gate(o, g, w, tiers, out=y)

    n = max(args.steps, 5)
    sep = timed(separate, n)
    fy = timed(lambda: gla.chunk_fwd_gated(q, k, v, gam, a, g, w, tiers, want_final_state=False), n)
    fyo = timed(lambda: gla.chunk_fwd_gated(q, k, v, gam, a, g, w, tiers, want_o=True,
                                            want_final_state=False), n)
    if gla.get_device_error() != 0:
        raise RuntimeError("device error")
    print(json.dumps(dict(part="fused", workload=f"GLA forward + output epilogue (4 tiers), B={Bf} "
                          "T=2048 H=16, bf16 q,k,v,g", separate_ms=sep, fused_y_ms=fy,
                          fused_y_and_o_ms=fyo, tokens_per_s_fused_y=Bf * T / (fy * 1e-3))),
          flush=True)
    return 0


def run_conv(args):
    """--part conv: the causal depth-wise conv + SiLU at the training shape (B=32, T=2048,
    D=3072, x bf16), forward and gradient, and one decode step over 1280 sequences x 24 layers
    of 3-input states."""
    import torch
    import gated_linear_attention_chunked_gb300 as gla
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gla.load()
    Dm = 3072
    gen = torch.Generator(device=dev)
    gen.manual_seed(55)
    Bc = args.batch
    x = torch.randn(Bc, T, Dm, generator=gen, device=dev).bfloat16()
    dy = torch.randn(Bc, T, Dm, generator=gen, device=dev)
    w = 0.5 * torch.randn(Dm, 4, generator=gen, device=dev)
    b = 0.1 * torch.randn(Dm, generator=gen, device=dev)
    init = torch.randn(Bc, 3, Dm, generator=gen, device=dev)
    y = torch.empty(Bc, T, Dm, device=dev)
    ws = torch.empty(gla.load().gla_conv_bwd_workspace_size(Bc, T, Dm), dtype=torch.uint8, device=dev)
    n_dec = args.n_seq * N_LAYERS
    st = torch.randn(n_dec, 3, Dm, generator=gen, device=dev)
    xd = torch.randn(n_dec, Dm, generator=gen, device=dev)
    yd = torch.empty_like(xd)
    stream = torch.cuda.current_stream()

    def timed(fn, n):
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    n = max(args.steps, 5)
    f_ms = timed(lambda: gla.conv_fwd(x, w, b, init, out=y), n)
    b_ms = timed(lambda: gla.conv_bwd(x, w, dy, b, init, workspace=ws), n)
    d_ms = timed(lambda: gla.conv_decode_step(st, xd, w, b, out=yd), n)
    if gla.get_device_error() != 0:
        raise RuntimeError("device error")
    el = Bc * T * Dm
    fb, bb = el * (2 + 4), el * (2 + 4 + 4)          # x bf16 + y | x + dy + dx
    db_ = n_dec * Dm * (3 * 4 * 2 + 4 + 4)            # state r+w, x, y
    pk = peaks()
    gbs = lambda byts, ms: byts / (ms * 1e-3) / 1e9
    print(json.dumps(dict(part="conv", workload=f"causal depth-wise conv k=4 + SiLU, B={Bc} T=2048 "
                          f"D=3072 (x bf16), decode over {args.n_seq} x 24 states", fwd_ms=f_ms,
                          fwd_gbs=gbs(fb, f_ms), fwd_frac_hbm=gbs(fb, f_ms) / pk["hbm"], bwd_ms=b_ms,
                          bwd_gbs=gbs(bb, b_ms), bwd_frac_hbm=gbs(bb, b_ms) / pk["hbm"],
                          decode_ms=d_ms, decode_gbs=gbs(db_, d_ms),
                          decode_frac_hbm=gbs(db_, d_ms) / pk["hbm"], peak_source=pk["src"])),
          flush=True)
    return 0


def run_head_norm(args):
    """--part norm: the output epilogue (Head RMSNorm per decay tier, SiLU(g) gate) and its
    gradient at the training shape B=32, T=2048, H=16, 4 tiers; o, dy fp32, g bf16."""
    import torch
    import gated_linear_attention_chunked_gb300 as gla
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gla.load()
    n_tok, tiers = args.batch * T, 4
    gen = torch.Generator(device=dev)
    gen.manual_seed(99)
    o = torch.randn(n_tok, H, DV, generator=gen, device=dev)
    g = torch.randn(n_tok, H, DV, generator=gen, device=dev).bfloat16()
    dy = torch.randn(n_tok, H, DV, generator=gen, device=dev)
    w = 1.0 + 0.2 * torch.randn(tiers, DV, generator=gen, device=dev)
    y = torch.empty_like(o)
    ws = torch.empty(gla.head_norm_gate_bwd_workspace_size(n_tok, H), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def timed(fn, n):
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    n = max(args.steps, 5)
    f_ms = timed(lambda: gla.head_norm_gate(o, g, w, tiers, out=y), n)
    b_ms = timed(lambda: gla.head_norm_gate_bwd(dy, o, g, w, tiers, workspace=ws), n)
    if gla.get_device_error() != 0:
        raise RuntimeError("device error")
    rows = n_tok * H
    fb = rows * (DV * 4 + DV * 2 + DV * 4)               # o, g in; y out
    bb = rows * (DV * 4 + DV * 4 + DV * 2 + 2 * DV * 4)  # dy, o, g in; d_o, dg out
    pk = peaks()
    print(json.dumps(dict(part="norm", workload=f"head RMSNorm (4 tiers) + SiLU gate, B={args.batch} "
                          "T=2048 H=16: o, dy fp32, g bf16", fwd_ms=f_ms, fwd_gbs=fb / (f_ms * 1e-3) / 1e9,
                          fwd_frac_hbm=fb / (f_ms * 1e-3) / 1e9 / pk["hbm"], bwd_ms=b_ms,
                          bwd_gbs=bb / (b_ms * 1e-3) / 1e9,
                          bwd_frac_hbm=bb / (b_ms * 1e-3) / 1e9 / pk["hbm"],
                          peak_source=pk["src"])), flush=True)
    return 0


def run_paged_decode(args):
    """--part paged: one decode step over the serving pool (1280 pages x 24 layers x 16 heads
    of 96x192 fp32 states) for an active set of 1024 sequences in shuffled page order, through
    gla_decode_step_paged."""
    import torch
    import gated_linear_attention_chunked_gb300 as gla
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gla.load()
    n_pages = args.n_seq
    n_act = n_pages * 4 // 5
    gen = torch.Generator(device=dev)
    gen.manual_seed(777)
    pool = torch.randn(n_pages, N_LAYERS, H, DK, DV, generator=gen, device=dev) * 0.05
    page = torch.randperm(n_pages, generator=gen, device=dev)[:n_act].to(torch.int32)
    q = torch.randn(n_act, N_LAYERS, H, DK, generator=gen, device=dev) * DK ** -0.5
    k = torch.randn(n_act, N_LAYERS, H, DK, generator=gen, device=dev)
    v = torch.randn(n_act, N_LAYERS, H, DV, generator=gen, device=dev)
    a = torch.randn(N_LAYERS, H, DK, generator=gen, device=dev) * 0.02
    gam = gla.decay_schedule(H).to(dev)
    o = torch.empty(n_act, N_LAYERS, H, DV, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        gla.decode_step_paged(pool, page, q, k, v, gam, a, out=o)
    n = max(args.steps, 5)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        gla.decode_step_paged(pool, page, q, k, v, gam, a, out=o)
    e1.record(stream)
    torch.cuda.synchronize()
    if gla.get_device_error() != 0:
        raise RuntimeError("device error")
    ms = e0.elapsed_time(e1) / n
    byts = n_act * N_LAYERS * H * DEC_BYTES_STATE
    pk = peaks()
    print(json.dumps(dict(part="paged", workload=f"paged decode, {n_act} active of {n_pages} pages "
                          "x 24 x 16 fp32 states, shuffled page order", ms=ms, gbs=byts / (ms * 1e-3) / 1e9,
                          frac_hbm=byts / (ms * 1e-3) / 1e9 / pk["hbm"], peak_source=pk["src"])),
          flush=True)
    return 0


def run_shard(args):
    """--part shard: what one rank runs when the long prefill (B=2, T=--long-t, H=16, bf16,
    initial state) is cut into R consecutive slices across R GPUs (--shard-ranks), measured on
    this GPU: the slice's state sum, the link of the gathered sums into the state entering the
    slice, the forward on the slice; then the adjoint sum, the reverse link and the backward.
    The last rank is timed (its forward link walks every slice before it).  The all-gather of
    the sums between those steps (B*H*73,728 B per rank each way) and the all-reduce of d_aug
    are not run: one GPU, so no multi-GPU time exists; the gathered sums are stand-ins of the
    right shape."""
    import torch
    import gated_linear_attention_chunked_gb300 as gla
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gla.load()
    R, Bl, Tl = args.shard_ranks, 2, args.long_t
    if R < 2 or Tl % R:
        raise SystemExit("--shard-ranks must be >= 2 and divide --long-t")
    Ts, r = Tl // R, R - 1
    gen = torch.Generator(device=dev)
    gen.manual_seed(4322)
    rn = lambda *sh, std=1.0: torch.randn(*sh, generator=gen, device=dev) * std
    q = rn(Bl, Ts, H, DK, std=DK ** -0.5).bfloat16()
    k = rn(Bl, Ts, H, DK).bfloat16()
    v = rn(Bl, Ts, H, DV).bfloat16()
    dO = rn(Bl, Ts, H, DV).bfloat16()
    init = rn(Bl, H, DK, DV, std=0.01)
    dfin = rn(Bl, H, DK, DV, std=0.01)
    a = rn(H, DK, std=0.02)
    gam = gla.decay_schedule(H).to(dev)
    U_all = rn(R, Bl, H, DK, DV, std=0.01)   # the all-gather's result (stand-ins)
    Ua_all = rn(R, Bl, H, DK, DV, std=0.01)
    lens = [Ts] * R
    s_in = torch.empty(Bl, H, DK, DV, device=dev)
    a_out = torch.empty(Bl, H, DK, DV, device=dev)
    o = torch.empty(Bl, Ts, H, DV, device=dev)
    fin = torch.empty(Bl, H, DK, DV, device=dev)
    gate = torch.empty(Bl, H, Ts, device=dev)
    ws_f = torch.empty(max(gla.chunk_fwd_workspace_size(Bl, Ts, H, gla.GLA_BF16), 256),
                       dtype=torch.uint8, device=dev)
    ws_b = torch.empty(max(gla.chunk_bwd_workspace_size(Bl, Ts, H, gla.GLA_BF16), 256),
                       dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    steps = {
        "fwd_state_sum": lambda: gla.chunk_state_sum(k, v, gam, out=U_all[r]),
        "fwd_link": lambda: gla.state_link(U_all, lens, r, gam, init, out=s_in),
        "fwd_slice": lambda: gla.chunk_fwd(q, k, v, gam, a, s_in, out=o, final_state=fin,
                                           gate=gate, workspace=ws_f),
        "bwd_adjoint_sum": lambda: gla.chunk_adjoint_sum(q, dO, gam, out=Ua_all[r]),
        "bwd_link": lambda: gla.state_link(Ua_all, lens, r, gam, dfin, reverse=True, out=a_out),
        "bwd_slice": lambda: gla.chunk_bwd(q, k, v, gam, a, dO, s_in, a_out, gate=gate,
                                           workspace=ws_b),
    }
    n = max(args.steps, 10)
    ms = {}
    for name, fn in steps.items():
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms[name] = e0.elapsed_time(e1) / n
    if gla.get_device_error() != 0:
        raise RuntimeError("device error in the sharded steps")
    f_ms = ms["fwd_state_sum"] + ms["fwd_link"] + ms["fwd_slice"]
    b_ms = ms["bwd_adjoint_sum"] + ms["bwd_link"] + ms["bwd_slice"]
    print(json.dumps(dict(
        part="shard", workload=f"long prefill B={Bl} T={Tl} H={H} bf16 cut into {R} slices of "
        f"{Ts} tokens, one per rank; rank {r} timed on one GPU without the exchange",
        ranks=R, slice_tokens=Ts, ms=ms, fwd_rank_ms=f_ms, bwd_rank_ms=b_ms,
        exchange_bytes_per_rank=Bl * H * DK * DV * 4,
        fwd_tokens_per_s_all_ranks_without_exchange=R * Bl * Ts / (f_ms * 1e-3),
        bwd_tokens_per_s_all_ranks_without_exchange=R * Bl * Ts / (b_ms * 1e-3),
        note="unmeasured: the all-gather and the d_aug all-reduce (one GPU per run)")),
        flush=True)
    return 0


def run_long_prefill(args):
    """--part long: the long-context prefill forward (B=2, T=131072, H=16, bf16, initial state
    ~ N(0, 0.01)), through the public API with its workspace (pairs cut into parts) and, for
    comparison, without one (one serial chunk scan per pair); then the backward of the same
    shape both ways."""
    import torch
    import gated_linear_attention_chunked_gb300 as gla
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = gla.load()
    gla.set_pass_overlap(args.pass_overlap)
    gla.set_split_parts(args.split_parts)
    Bl, Tl = 2, args.long_t
    gen = torch.Generator(device=dev)
    gen.manual_seed(4321)
    rn = lambda *sh, std=1.0: torch.randn(*sh, generator=gen, device=dev) * std
    q = rn(Bl, Tl, H, DK, std=DK ** -0.5).bfloat16()
    k = rn(Bl, Tl, H, DK).bfloat16()
    v = rn(Bl, Tl, H, DV).bfloat16()
    init = rn(Bl, H, DK, DV, std=0.01)
    a = rn(H, DK, std=0.02)
    gam = gla.decay_schedule(H).to(dev)
    o = torch.empty(Bl, Tl, H, DV, device=dev)
    fin = torch.empty(Bl, H, DK, DV, device=dev)
    gl = torch.empty(Bl, H, Tl, device=dev)  # the gate, saved for the backward below
    nws = gla.chunk_fwd_workspace_size(Bl, Tl, H, gla.GLA_BF16)
    ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call(w, nb):
        rc = lib.gla_chunk_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), gla.GLA_BF16,
                               gam.data_ptr(), a.data_ptr(), init.data_ptr(), o.data_ptr(),
                               fin.data_ptr(), gl.data_ptr(), None, 0, w, nb, Bl, Tl, H, DK, DV,
                               stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(gla.status_string(rc))

    def timed(w, nb, n):
        for _ in range(args.warmup):
            call(w, nb)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            call(w, nb)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    seg_ms = timed(ws.data_ptr(), nws, max(args.steps, 5))
    ser_ms = timed(None, 0, 3)
    plan_f = gla.split_plan(Bl, Tl, H, False, torch.cuda.get_device_properties(dev).multi_processor_count)

    # the backward of the same shape: with the workspace that lets pairs be cut, and with only
    # the part it requires
    dO = rn(Bl, Tl, H, DV).bfloat16()
    dq, dk = torch.empty(Bl, Tl, H, DK, device=dev), torch.empty(Bl, Tl, H, DK, device=dev)
    dv, dinit = torch.empty(Bl, Tl, H, DV, device=dev), torch.empty(Bl, H, DK, DV, device=dev)
    d_a = torch.empty(H, DK, device=dev)
    nwb = gla.chunk_bwd_workspace_size(Bl, Tl, H, gla.GLA_BF16)
    wsb = torch.empty(nwb, dtype=torch.uint8, device=dev)
    nwb_min = 256 * ((Bl * H * DK * 4 + 255) // 256)  # the d_aug partial sums only

    def call_b(nb):
        rc = lib.gla_chunk_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), gla.GLA_BF16,
                               gam.data_ptr(), a.data_ptr(), init.data_ptr(), dO.data_ptr(), None,
                               gl.data_ptr(), None, 0, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                               d_a.data_ptr(), dinit.data_ptr(), wsb.data_ptr(), nb, Bl, Tl, H,
                               DK, DV, stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(gla.status_string(rc))

    def timed_b(nb, n):
        call_b(nb)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            call_b(nb)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    bwd_ms = timed_b(nwb, 3)
    bwd_ser_ms = timed_b(nwb_min, 2)
    n_sm_l = torch.cuda.get_device_properties(dev).multi_processor_count
    plan_b = gla.split_plan(Bl, Tl, H, 1, n_sm_l)

    # the same shape as a training step: the forward also saves its state copies (1.2 GB here)
    # and the backward reads them, so its dq part needs no state scan
    saved = torch.empty(gla.chunk_saved_states_size(Bl, Tl, H), dtype=torch.uint8, device=dev)
    gla.chunk_fwd(q, k, v, gam, a, init, out=o, final_state=fin, gate=gl, saved_states=saved,
                  workspace=ws)

    def train_bwd():
        gla.chunk_bwd(q, k, v, gam, a, dO, init, gate=gl, saved_states=saved, workspace=wsb)

    train_bwd()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(3):
        train_bwd()
    e1.record(stream)
    torch.cuda.synchronize()
    bwd_saved_ms = e0.elapsed_time(e1) / 3
    if gla.get_device_error() != 0:
        raise RuntimeError("device error")
    byts = Bl * Tl * H * FWD_BYTES_TH
    pk = peaks()
    print(json.dumps(dict(part="long", workload=f"long prefill fwd B=2 T={Tl} H=16 bf16 in, fp32 out",
                          ms=seg_ms, tokens_per_s=Bl * Tl / (seg_ms * 1e-3),
                          gbs=byts / (seg_ms * 1e-3) / 1e9, frac_hbm=byts / (seg_ms * 1e-3) / 1e9 / pk["hbm"],
                          peak_source=pk["src"], workspace_bytes=nws, serial_ms=ser_ms,
                          plan_fwd=plan_f, bwd_ms=bwd_ms, bwd_serial_ms=bwd_ser_ms,
                          bwd_tokens_per_s=Bl * Tl / (bwd_ms * 1e-3), plan_bwd=plan_b,
                          bwd_saved_states_ms=bwd_saved_ms,
                          plan_bwd_saved_states=gla.split_plan(Bl, Tl, H, 2, n_sm_l))), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-saved-states", dest="saved_states", action="store_false",
                    help="the training step without the forward's saved state copies")
    ap.add_argument("--no-pass-overlap", dest="pass_overlap", action="store_false",
                    help="segment passes before the whole pairs on the caller's stream")
    ap.add_argument("--split-parts", type=int, default=0,
                    help="gla_set_split_parts: 0 automatic, 1 never cut, p >= 2 forced")
    ap.add_argument("--cpu-configs", action="store_true",
                    help="time the fp64 CPU oracle on every workload (no GPU work)")
    ap.add_argument("--cpu-seqs", type=int, default=32,
                    help="sequences of the training workload the CPU oracle baseline times")
    ap.add_argument("--part", choices=["all", "fwd", "bwd", "decode", "long", "paged", "norm", "conv", "fused", "shard"], default="all",
                    help="time one call alone (smaller profiling cases); the default is the "
                         "whole hot path")
    ap.add_argument("--batch", type=int, default=B, help="sequences of the training shape")
    ap.add_argument("--n-seq", type=int, default=N_SEQ, help="sequences of the serving pool")
    ap.add_argument("--long-t", type=int, default=131072, help="tokens of the long prefill (--part long, shard)")
    ap.add_argument("--shard-ranks", type=int, default=8,
                    help="--part shard: ranks the long prefill is cut across (one slice each)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.part != "all":
        args.no_e2e = True
    if args.part != "all" or args.batch != B or args.n_seq != N_SEQ:
        args.no_cpu_baseline = True  # the oracle's samples are of the default workload
    if args.gpus > 1 and world == 1:
        print("bench.py: for --gpus N > 1 launch with torch.distributed.run (one rank per GPU)",
              file=sys.stderr)
        return 2
    if args.cpu_configs:
        return run_cpu_configs(args) if rank == 0 else 0
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.part == "long":
        return run_long_prefill(args) if rank == 0 else 0
    if args.part == "paged":
        return run_paged_decode(args) if rank == 0 else 0
    if args.part == "norm":
        return run_head_norm(args) if rank == 0 else 0
    if args.part == "conv":
        return run_conv(args) if rank == 0 else 0
    if args.part == "fused":
        return run_fused(args) if rank == 0 else 0
    if args.part == "shard":
        return run_shard(args) if rank == 0 else 0
    return run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
